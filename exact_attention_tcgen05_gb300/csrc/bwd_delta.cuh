// bwd_delta.cuh - backward preprocess: D_i = sum_c dO_ic * O_ic for every row
// ("Triton 05: Flash Attention", section Softmax Gradient, and section 3단계 커널 구조,
// [1단계] Preprocess 커널: in O, dO (bh, N, d), out D (bh * N)).
//
// Pure streaming work (reads 4 bytes per element pair, writes 4 bytes per row), so it is
// bound by HBM bandwidth: each group of d/8 lanes reads one row with 16-byte vector
// loads (a warp touches 512 contiguous bytes per tensor per load), every lane keeps
// several rows in flight, partial dot products are reduced with warp shuffles, and the
// grid is a whole number of waves over the 152 SMs (grid-stride loop).
#pragma once

#include "common.cuh"

namespace attn {

constexpr int kDeltaThreads = 256;
constexpr int kDeltaUnroll = 4;

template <bool BF16>
__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 fa, fb;
    if constexpr (BF16) {
      fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[i]));
      fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bv[i]));
    } else {
      fa = __half22float2(*reinterpret_cast<const __half2*>(&av[i]));
      fb = __half22float2(*reinterpret_cast<const __half2*>(&bv[i]));
    }
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
  return acc;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// rows = B*H*N; o, dO: rows x D 16-bit; delta: rows f32, row r at delta[r].
// Packed batch (PACKED): rows = total*H in [total, H] order, and the D of row
// r = t*H + h goes to delta[h*total + t] (the [H, total] layout of lse).
template <int D, bool BF16, bool PACKED>
__global__ void __launch_bounds__(kDeltaThreads)
    attn_bwd_delta_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dO,
                          float* __restrict__ delta, long long rows, int heads,
                          long long total, int n16) {
  // n16: 16-byte pieces per row (head dimension / 8, at most D / 8); lanes past it add 0.
  constexpr int kLanesPerRow = D / 8;              // 16-byte chunks per row
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;  // rows one warp covers per load
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow;
  const int part = lane % kLanesPerRow;
  const long long warp_g = ((long long)blockIdx.x * kDeltaThreads + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * kDeltaThreads) >> 5;
  constexpr int kRowsPerStep = kRowsPerWarp * kDeltaUnroll;
  for (long long r0 = warp_g * kRowsPerStep; r0 < rows; r0 += nwarps * kRowsPerStep) {
    uint4 a[kDeltaUnroll], b[kDeltaUnroll];
#pragma unroll
    for (int u = 0; u < kDeltaUnroll; ++u) {
      const long long row = r0 + u * kRowsPerWarp + sub;
      if (row < rows && part < n16) {
        a[u] = ld_stream(o + row * n16 + part);
        b[u] = ld_stream(dO + row * n16 + part);
      } else {
        a[u] = make_uint4(0, 0, 0, 0);
        b[u] = a[u];
      }
    }
#pragma unroll
    for (int u = 0; u < kDeltaUnroll; ++u) {
      float acc = dot8<BF16>(a[u], b[u]);
#pragma unroll
      for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const long long row = r0 + u * kRowsPerWarp + sub;
      if (part == 0 && row < rows)
        delta[PACKED ? (row % heads) * total + row / heads : row] = acc;
    }
  }
}

}  // namespace attn
