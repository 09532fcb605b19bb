// common.cuh - shapes and tile geometry shared by the attention kernels.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"
#include "varlen.h"

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
  kWaitFwdDrain, kWaitFwdX, kWaitFwdQEmpty, kWaitFwdOFree,
  kWaitFwdPeer,  // CTA pairs: rank 1's copies (forwarded to rank 0)
  kWaitFwdExit,  // CTA pairs: the exit handshake
  kWaitDqQ = 0x21, kWaitDqK, kWaitDqV, kWaitDqEmpty, kWaitDqS, kWaitDqDP, kWaitDqDS,
  kWaitDqDone, kWaitDqDrain, kWaitDqSC, kWaitDqQFree, kWaitDqAccFree,
  kWaitDkvKV = 0x31, kWaitDkvQ, kWaitDkvDO, kWaitDkvEmpty, kWaitDkvS, kWaitDkvDP,
  kWaitDkvP, kWaitDkvDS, kWaitDkvDone, kWaitDkvDrain, kWaitDkvStats, kWaitDkvKVFree,
  kWaitDkvAccFree,
  kWaitDecFull = 0x41, kWaitDecDrain,
  kErrPairTmem = kStatusPairTmem,  // CTA pairs: the two tensor-memory allocations differ
  kErrSeqlens = kStatusBadSeqlens,  // a packed batch's cu_seqlens hold a bad sequence
  kErrSmemAlign = kStatusSmemAlign  // dynamic shared memory not 1024-byte aligned
};

// Bound of the waits that let a CTA's own in-flight work finish before it releases shared
// or tensor memory (copies it started, MMAs it issued). Deliberately independent of the
// configurable pipeline limit: after a pipeline wait gives up, these must still see that
// work complete (microseconds), or memory could be released under it.
constexpr unsigned long long kDrainLimit = 1ull << 31;

// Where the rows of one (sequence, head) slice live.
//   dense:  TMA coordinates (col, row, bh) of a [B*H, N, d] map; element offset of row r
//           = bh*N*d + r*d.
//   packed: TMA coordinates (col, h, start + r) of a [total, H, d] map; element offset
//           of row r = ((start + r)*H + h)*d.
struct SliceRows {
  int nq, nk;            // query and key rows of the slice
  int off;               // nk - nq: causal key j is visible to query i iff j <= i + off
  int q_start, k_start;  // first token of the sequence (packed) or 0
  int tma_bh;            // bh (dense) or h (packed)
  bool packed;
  size_t q_elem0, k_elem0;  // element offset of row 0 of the q-like / k-like tensors
  size_t row_elems;         // elements between consecutive rows
  size_t stat0;             // index of row 0 in lse and D
};

// Fills `s` for slice bh; D is the head dimension of the tensors (elements per row). Dense
// (PACKED = false): the whole-call sizes N, Nk. Packed:
// reads the slice's sequence bounds and checks them (in range, not longer than the grid
// covers, and every query row sees a key); a malformed sequence records kErrSeqlens and
// returns false. The layout is a template parameter so that the dense kernels carry no
// trace of the packed addressing.
template <bool PACKED>
__device__ __forceinline__ bool slice_rows(const Varlen& vl, int bh, int N, int Nk, int D,
                                           bool causal, SliceRows& s) {
  if constexpr (!PACKED) {
    s.nq = N;
    s.nk = Nk;
    s.q_start = s.k_start = 0;
    s.tma_bh = bh;
    s.packed = false;
    s.q_elem0 = (size_t)bh * N * D;
    s.k_elem0 = (size_t)bh * Nk * D;
    s.row_elems = (size_t)D;
    s.stat0 = (size_t)bh * N;
  } else {
    const int b = bh / vl.H, h = bh % vl.H;
    const int q0 = vl.cu_q[b], q1 = vl.cu_q[b + 1];
    const int k0 = vl.cu_k[b], k1 = vl.cu_k[b + 1];
    const bool bad = q0 < 0 || q1 < q0 || q1 > vl.total_q || k0 < 0 || k1 < k0 ||
                     k1 > vl.total_k || q1 - q0 > vl.max_q || k1 - k0 > vl.max_k ||
                     (q1 > q0 && (k1 == k0 || (causal && k1 - k0 < q1 - q0)));
    if (bad) {
      record_timeout(kErrSeqlens);
      return false;
    }
    s.nq = q1 - q0;
    s.nk = k1 - k0;
    s.q_start = q0;
    s.k_start = k0;
    s.tma_bh = h;
    s.packed = true;
    s.q_elem0 = ((size_t)q0 * vl.H + h) * D;
    s.k_elem0 = ((size_t)k0 * vl.H + h) * D;
    s.row_elems = (size_t)vl.H * D;
    s.stat0 = (size_t)h * vl.total_q + q0;
  }
  s.off = s.nk - s.nq;
  return true;
}

// TMA copy of one [128 rows x 64 cols] box of a slice, starting at slice row `row`
// (`keys`: a k-like tensor), in the slice's layout (see SliceRows).
template <bool PACKED>
__device__ __forceinline__ void tma_load_rows(void* dst, const CUtensorMap* map, uint64_t* bar,
                                              int col, int row, const SliceRows& s, bool keys) {
  if constexpr (PACKED)
    tma_load_3d(dst, map, bar, col, s.tma_bh, (keys ? s.k_start : s.q_start) + row);
  else
    tma_load_3d(dst, map, bar, col, row, s.tma_bh);
}

// Head dimensions other than the kernels' own (64 or 128): a tensor row of dh elements is
// loaded into a D-column tile whose columns past dh read as zero (TMA fills them, or the
// row copies below do), so every product sees exact zeros there; only the first dh columns
// are stored. These give the number of valid 16-byte pieces (8 columns each).
__device__ __forceinline__ int valid16(int dh, int col0, int max16) {
  const int v = (dh - col0) / 8;
  return v < 0 ? 0 : (v > max16 ? max16 : v);
}

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

// Copies one 16-bit row of n16 16-byte pieces from global memory (zeros past them, and
// everywhere when src is null) into tensor-memory columns [t_col, t_col + D/2) of this
// thread's lane as packed pairs (the layout of an A operand read from tensor memory). Every
// lane of the warp calls it (the TMEM store is warp-collective).
template <int D>
__device__ __forceinline__ void copy_row_to_tmem(const uint8_t* src, uint32_t t_col,
                                                 int n16 = D / 8) {
  // Every load of the row is issued before the first tensor-memory store (the stores are
  // ordering points for the compiler), so the row costs one memory latency, not D / 64.
  uint32_t r[D / 2];
#pragma unroll
  for (int k = 0; k < D / 8; ++k) {
    const uint4 v = (src && k < n16) ? *reinterpret_cast<const uint4*>(src + k * 16)
                                     : make_uint4(0, 0, 0, 0);
    r[4 * k] = v.x;
    r[4 * k + 1] = v.y;
    r[4 * k + 2] = v.z;
    r[4 * k + 3] = v.w;
  }
#pragma unroll
  for (int c = 0; c < D / 64; ++c)
    tmem_st32(t_col + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&r[32 * c]));
}

// D[128 x 64] = A B^T over 256 columns, both K-major with 128-byte swizzle: A a [128 x 256]
// tile (four 16 KiB boxes of 64 columns), B a [64 x 256] block (four 8 KiB boxes), 16
// steps of 16 columns (the score products of the kernels for head dims above 128).
// Descriptors built once by the caller; the start-address field is advanced by byte
// offset / 16.
__device__ __forceinline__ void issue_rowdot_wide(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < 256 / 16; ++kk) {
    const uint32_t a_off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
    const uint32_t b_off = ((kk >> 2) * (kBoxBytes / 2) + (kk & 3) * 32) >> 4;
    mma_ss(d_tmem, a_desc + a_off, b_desc + b_off, idesc, kk > 0 ? 1u : 0u);
  }
}

// D[128 x 64] = A B^T over 256 columns with A in tensor memory (16-bit pairs from column
// a_tmem, 128 columns) and B a K-major [64 x 256] block (four 8 KiB boxes).
__device__ __forceinline__ void issue_rowdot_ts_wide(uint32_t d_tmem, uint32_t a_tmem,
                                                     uint64_t b_desc, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < 256 / 16; ++kk) {
    const uint32_t b_off = ((kk >> 2) * (kBoxBytes / 2) + (kk & 3) * 32) >> 4;
    mma_ts(d_tmem, a_tmem + kk * 8, b_desc + b_off, idesc, kk > 0 ? 1u : 0u);
  }
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
