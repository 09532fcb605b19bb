// kernels_dkv.cu - instantiation and launch of the backward dK/dV kernel.
#include "bwd_dkv.cuh"
#include "launch.h"

namespace attn {

template <int D, bool BF16>
static cudaError_t launch_dkv_t(const Maps& m, const Shape& s, const void* q, const void* k,
                                const void* v, const void* d_o, const float* lse,
                                const float* delta, void* dk, void* dv, cudaStream_t st) {
  using C = DkvCfg<D>;
  // d = 64: K_j, V_j in tensor memory when a key block meets about eight or more query
  // blocks (the one-time row copy costs more than it saves on shorter work).
  const bool kv_tmem = D == 64 && (s.causal ? s.N >= 2048 : s.N >= 1024);
  auto kern = s.vl.cu_q != nullptr
                  ? (kv_tmem ? attn_bwd_dkv_kernel<D, BF16, true, D == 64>
                             : attn_bwd_dkv_kernel<D, BF16, true, false>)
                  : (kv_tmem ? attn_bwd_dkv_kernel<D, BF16, false, D == 64>
                             : attn_bwd_dkv_kernel<D, BF16, false, false>);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  BwdParams p;
  p.in_q = q;
  p.in_k = k;
  p.in_v = v;
  p.in_do = d_o;
  p.lse = lse;
  p.delta = delta;
  p.out0 = dk;
  p.out1 = dv;
  p.dh = s.d;
  p.N = s.N;
  p.Nk = s.Nk;
  p.vl = s.vl;
  p.causal = s.causal ? 1 : 0;
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  // One CTA per 128-key block (packed batches: of the longest sequence).
  dim3 grid((s.Nk + kTileN - 1) / kTileN, s.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(m.q, m.k, m.v, m.d_o, p);
  return cudaGetLastError();
}

cudaError_t launch_dkv(const Maps& m, const Shape& s, const void* q, const void* k,
                       const void* v, const void* d_o, const float* lse, const float* delta,
                       void* dk, void* dv, cudaStream_t st) {
  if (s.d > 64)
    return s.bf16 ? launch_dkv_t<128, true>(m, s, q, k, v, d_o, lse, delta, dk, dv, st)
                  : launch_dkv_t<128, false>(m, s, q, k, v, d_o, lse, delta, dk, dv, st);
  return s.bf16 ? launch_dkv_t<64, true>(m, s, q, k, v, d_o, lse, delta, dk, dv, st)
                : launch_dkv_t<64, false>(m, s, q, k, v, d_o, lse, delta, dk, dv, st);
}

ATTN_DEFINE_STATUS_READER(status_dkv)

}  // namespace attn
