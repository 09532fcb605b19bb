// varlen.h - description of a packed variable-length batch, shared by the host launch
// code and the kernels.
//
// "FlashAttentionを1から — 計算を増やして速くする逆説", section 現場ではこう使う: padding
// sequences of different lengths to the longest one pays for the padded positions; the
// variable-length interface takes the sequence boundaries as cu_seqlens instead. Here
// the B sequences lie one after another along the token axis: q-like tensors are
// [total_q, H, d], k-like tensors [total_k, H, d], lse and D [H, total_q]; sequence b owns
// query tokens cu_q[b] .. cu_q[b+1]-1 and key tokens cu_k[b] .. cu_k[b+1]-1.
#pragma once

namespace attn {

// Status-word code of a kernel that found a malformed sequence in cu_seqlens.
constexpr int kStatusBadSeqlens = 0x7E;
// Status codes of a kernel that found its launch unusable and did nothing: the two
// tensor-memory allocations of a CTA pair at different addresses; dynamic shared memory
// not 1024-byte aligned.
constexpr int kStatusPairTmem = 0x7D;
constexpr int kStatusSmemAlign = 0x7F;

struct Varlen {
  const int* cu_q;  // [B + 1] cumulative query lengths in device memory; null = dense
  const int* cu_k;  // [B + 1] cumulative key lengths in device memory
  int H;
  int total_q, total_k;
  int max_q, max_k;  // longest query / key sequence: the grid covers this many rows
};

}  // namespace attn
