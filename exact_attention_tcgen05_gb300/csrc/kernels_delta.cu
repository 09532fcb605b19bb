// kernels_delta.cu - instantiation and launch of the backward preprocess (D) kernel.
#include "bwd_delta.cuh"
#include "launch.h"

namespace attn {

static int sm_count_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

template <int D, bool BF16>
static cudaError_t launch_delta_t(const Shape& s, const void* o, const void* dO, float* delta,
                                  cudaStream_t st) {
  const bool packed = s.vl.cu_q != nullptr;
  const long long rows = packed ? (long long)s.vl.total_q * s.vl.H : (long long)s.BH * s.N;
  constexpr int kRowsPerBlockStep = (kDeltaThreads / 32) * (32 / (D / 8)) * kDeltaUnroll;
  const long long want = (rows + kRowsPerBlockStep - 1) / kRowsPerBlockStep;
  const int resident = 2048 / kDeltaThreads;  // blocks per SM at full occupancy
  const long long cap = (long long)sm_count_current() * resident;
  const int blocks = (int)(want < cap ? want : cap);
  auto kern = packed ? attn_bwd_delta_kernel<D, BF16, true> : attn_bwd_delta_kernel<D, BF16, false>;
  kern<<<blocks, kDeltaThreads, 0, st>>>(reinterpret_cast<const uint4*>(o),
                                         reinterpret_cast<const uint4*>(dO), delta, rows,
                                         packed ? s.vl.H : 0,
                                         packed ? (long long)s.vl.total_q : 0, s.d / 8);
  return cudaGetLastError();
}

cudaError_t launch_delta(const Shape& s, const void* o, const void* dO, float* delta,
                         cudaStream_t st) {
  if (s.d > 128) return s.bf16 ? launch_delta_t<256, true>(s, o, dO, delta, st)
                                 : launch_delta_t<256, false>(s, o, dO, delta, st);
  if (s.d > 64) return s.bf16 ? launch_delta_t<128, true>(s, o, dO, delta, st)
                                : launch_delta_t<128, false>(s, o, dO, delta, st);
  return s.bf16 ? launch_delta_t<64, true>(s, o, dO, delta, st)
                : launch_delta_t<64, false>(s, o, dO, delta, st);
}

ATTN_DEFINE_STATUS_READER(status_delta)

}  // namespace attn
