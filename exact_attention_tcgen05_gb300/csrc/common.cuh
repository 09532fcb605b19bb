// common.cuh - shapes and tile geometry shared by the attention kernels.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace attn {

constexpr int kTileM = 128;           // query rows per MMA tile (TMEM lanes)
constexpr int kTileN = 128;           // keys per key/value block
constexpr int kBoxCols = 64;          // 16-bit elements per 128-byte swizzled row
constexpr int kBoxBytes = 128 * 128;  // one [128 rows x 64 cols] 16-bit box = 16 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Codes recorded in the status word when a bounded wait gives up (kernel * 16 + site).
enum WaitSite : int {
  kWaitFwdQ = 0x11, kWaitFwdK, kWaitFwdV, kWaitFwdEmpty, kWaitFwdS, kWaitFwdP, kWaitFwdO,
  kWaitFwdDrain, kWaitFwdX,
  kWaitDqQ = 0x21, kWaitDqK, kWaitDqV, kWaitDqEmpty, kWaitDqS, kWaitDqDP, kWaitDqDS,
  kWaitDqDone, kWaitDqDrain, kWaitDqSC,
  kWaitDkvKV = 0x31, kWaitDkvQ, kWaitDkvDO, kWaitDkvEmpty, kWaitDkvS, kWaitDkvDP,
  kWaitDkvP, kWaitDkvDS, kWaitDkvDone, kWaitDkvDrain, kWaitDkvStats,
  kWaitDecFull = 0x41, kWaitDecDrain,
  kErrSmemAlign = 0x7F  // dynamic shared memory not 1024-byte aligned (kernel skipped)
};

// Bound of the waits that let a CTA's own in-flight work finish before it releases shared
// or tensor memory (copies it started, MMAs it issued). Deliberately independent of the
// configurable pipeline limit: after a pipeline wait gives up, these must still see that
// work complete (microseconds), or memory could be released under it.
constexpr unsigned long long kDrainLimit = 1ull << 31;

// Rounds a shared-memory pointer up to 1024 bytes (the swizzle-atom alignment).
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

// Warp-uniform bounded wait: every lane waits; the result is true only if all did.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit,
                                          volatile int* abort, int where) {
  const bool ok = mbar_wait(bar, parity, limit, abort, where);
  return __all_sync(0xffffffffu, ok);
}

// Warp-uniform bounded poll (non-suspending test_wait in every lane): for the converged
// MMA-issuing warps.
__device__ __forceinline__ bool warp_poll(uint64_t* bar, uint32_t parity, uint64_t limit,
                                          volatile int* abort, int where) {
  const bool ok = mbar_poll(bar, parity, limit, abort, where);
  return __all_sync(0xffffffffu, ok);
}

// A operand in tensor memory whose 16-bit pairs sit in two halves: columns [0, 64) of A in
// [base, base + 32) and columns [64, 128) in [base + 64, base + 96). B is an MN-major
// [128 x d] tile in shared memory. D[128 x d] (+)= A B.
__device__ __forceinline__ void issue_tmem_a_split(uint32_t d_tmem, uint32_t a_tmem,
                                                   uint32_t b0, uint32_t idesc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 128 / 16; ++kk) {
    const uint32_t a_col = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;
    mma_ts(d_tmem, a_tmem + a_col, make_sdesc_sw128(b0 + kk * 2048, kBoxBytes, 1024), idesc,
           (acc || kk > 0) ? 1u : 0u);
  }
}

// A operand [128 x d] in tensor memory (16-bit pairs from column a_tmem) times a K-major
// B tile [128 x d] in shared memory: D[128 x 128] = A B^T.
template <int D>
__device__ __forceinline__ void issue_rowdot_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b0,
                                                uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
    mma_ts(d_tmem, a_tmem + kk * 8, make_sdesc_sw128(b0 + off, 16, 1024), idesc,
           kk > 0 ? 1u : 0u);
  }
}

// The two products above with the shared-memory descriptor of the B tile built once by
// the caller (make_sdesc_sw128 of the tile's first byte). The start-address field (bits
// 0-13, in 16-byte units) is advanced by adding byte offset / 16, which cannot carry out
// of the field for shared addresses below 256 KiB. Saves the single MMA-issuing thread
// the descriptor arithmetic of every k-step.
template <int D>
__device__ __forceinline__ void issue_rowdot_ts_d(uint32_t d_tmem, uint32_t a_tmem,
                                                  uint64_t b_desc, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
    mma_ts(d_tmem, a_tmem + kk * 8, b_desc + (off >> 4), idesc, kk > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ void issue_tmem_a_split_d(uint32_t d_tmem, uint32_t a_tmem,
                                                     uint64_t b_desc, uint32_t idesc,
                                                     bool acc) {
#pragma unroll
  for (int kk = 0; kk < 128 / 16; ++kk) {
    const uint32_t a_col = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;
    mma_ts(d_tmem, a_tmem + a_col, b_desc + ((kk * 2048) >> 4), idesc,
           (acc || kk > 0) ? 1u : 0u);
  }
}

// K-major x K-major product over the head dimension, D[128 x 128] = A[128 x d] B[128 x d]^T,
// with both shared-memory descriptors built once by the caller (see issue_rowdot_ts_d).
template <int D>
__device__ __forceinline__ void issue_rowdot_d(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
    mma_ss(d_tmem, a_desc + off, b_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

}  // namespace attn
