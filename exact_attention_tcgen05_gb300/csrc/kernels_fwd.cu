// kernels_fwd.cu - instantiation and launch of the forward kernel.
#include "fwd.cuh"
#include "launch.h"

namespace attn {

template <int D, bool BF16>
static cudaError_t launch_fwd_t(const Maps& m, const Shape& s, void* o, float* lse,
                                cudaStream_t st) {
  using C = FwdCfg<D>;
  auto kern = s.vl.cu_q != nullptr ? attn_fwd_kernel<D, BF16, true>
                                   : attn_fwd_kernel<D, BF16, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.N = s.N;
  p.Nk = s.Nk;
  p.causal = s.causal ? 1 : 0;
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  p.vl = s.vl;
  // Packed batches: s.N is the longest query sequence; CTAs past a sequence's end exit.
  dim3 grid((s.N + 2 * kTileM - 1) / (2 * kTileM), s.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(m.q, m.k, m.v, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const Maps& m, const Shape& s, void* o, float* lse, cudaStream_t st) {
  if (s.d == 128) return s.bf16 ? launch_fwd_t<128, true>(m, s, o, lse, st)
                                : launch_fwd_t<128, false>(m, s, o, lse, st);
  return s.bf16 ? launch_fwd_t<64, true>(m, s, o, lse, st)
                : launch_fwd_t<64, false>(m, s, o, lse, st);
}

ATTN_DEFINE_STATUS_READER(status_fwd)

}  // namespace attn
