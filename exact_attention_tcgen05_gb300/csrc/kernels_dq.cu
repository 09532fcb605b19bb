// kernels_dq.cu - instantiation and launch of the backward dQ kernel.
#include "bwd_dq.cuh"
#include "launch.h"

namespace attn {

template <int D, bool BF16>
static cudaError_t launch_dq_t(const Maps& m, const Shape& s, const void* q,
                               const void* d_o, const float* lse,
                               const float* delta, void* dq, cudaStream_t st) {
  using C = DqCfg<D>;
  auto kern = s.vl.cu_q != nullptr ? attn_bwd_dq_kernel<D, BF16, true>
                                   : attn_bwd_dq_kernel<D, BF16, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  BwdParams p;
  p.in_q = q;
  p.in_k = nullptr;
  p.in_v = nullptr;
  p.in_do = d_o;
  p.lse = lse;
  p.delta = delta;
  p.out0 = dq;
  p.out1 = nullptr;
  p.N = s.N;
  p.Nk = s.Nk;
  p.vl = s.vl;
  p.causal = s.causal ? 1 : 0;
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  // One CTA per 128-row query block (packed batches: of the longest sequence).
  dim3 grid((s.N + kTileM - 1) / kTileM, s.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(m.q, m.k, m.v, m.d_o, p);
  return cudaGetLastError();
}

cudaError_t launch_dq(const Maps& m, const Shape& s, const void* q, const void* d_o,
                       const float* lse, const float* delta,
                      void* dq, cudaStream_t st) {
  if (s.d == 128) return s.bf16 ? launch_dq_t<128, true>(m, s, q, d_o, lse, delta, dq, st)
                                : launch_dq_t<128, false>(m, s, q, d_o, lse, delta, dq, st);
  return s.bf16 ? launch_dq_t<64, true>(m, s, q, d_o, lse, delta, dq, st)
                : launch_dq_t<64, false>(m, s, q, d_o, lse, delta, dq, st);
}

ATTN_DEFINE_STATUS_READER(status_dq)

}  // namespace attn
