// launch.h - internal interface between the C ABI (attn_api.cu) and the translation
// units that hold the kernels. Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "varlen.h"

namespace attn {

// TMA descriptors of the [B*H, N, d] 16-bit tensors a kernel reads.
struct Maps {
  CUtensorMap q, k, v, d_o;
  // k read in [64-column x 64-row] boxes: the key halves of the CTA-pair forward, and the
  // 64-key blocks of the forward for head dims above 128 (encoded by the forward entry
  // points for d > 64)
  CUtensorMap k64;
  // v read in [64-column x 64-row] boxes: the forward and backward for head dims above 128
  // (encoded by the dense entry points for d > 128; k64 likewise for the backward)
  CUtensorMap v64;
  // q and dO read in [64-column x 64-row] boxes: the dK/dV passes of the backward for head
  // dims above 128 (encoded by the dense backward entry points for d > 128)
  CUtensorMap q64, do64;
  // o written in [64-column x 32-row] boxes: the persistent forward's staged epilogue at
  // d <= 64 (encoded by the dense forward entry point)
  CUtensorMap o;
  // dk, dv written in [64-column x 32-row] boxes: the persistent dK/dV kernel's staged
  // epilogue at d <= 64 (encoded by the dense backward entry points)
  CUtensorMap dk, dv;
  // dq written in unswizzled [32-column x 32-row] boxes: the persistent dQ kernel's staged
  // epilogue at d <= 64 (encoded by the dense backward entry points)
  CUtensorMap dq;
};

struct Shape {
  int BH, N, d;  // N: query rows per slice (N_q); packed batches: the longest sequence
  int Nk;        // key rows per slice (N_k); causal masking is bottom-right aligned
  bool bf16, causal;
  float scale;
  unsigned long long wait_limit;  // SM cycles one pipeline wait may take
  int stall = 0;  // failure tests: each kernel's copies are withheld (ATTN_TEST_STALL = 1)
  Varlen vl;     // packed variable-length batch; vl.cu_q == nullptr for dense tensors
  // Packed batches: HOST copies of vl.cu_q / vl.cu_k ([vl_b + 1] each), or null. Used only
  // to order the persistent kernels' work items (schedule.h); the kernels read the device
  // copies, and every item slot is processed whatever the host copies say.
  const int* host_cu_q = nullptr;
  const int* host_cu_k = nullptr;
  int vl_b = 0;  // sequences in the packed batch
};

// Query and key rows of slice bh (packed: of its sequence, from the host copies; a
// malformed entry counts as empty). Host only; for ordering work, never for addressing.
inline void slice_lengths(const Shape& s, int bh, int& nq, int& nk) {
  if (s.vl.cu_q == nullptr) {
    nq = s.N;
    nk = s.Nk;
    return;
  }
  const int b = bh / s.vl.H;
  nq = s.host_cu_q[b + 1] - s.host_cu_q[b];
  nk = s.host_cu_k[b + 1] - s.host_cu_k[b];
  if (nq < 0 || nq > s.vl.max_q || nk < 0 || nk > s.vl.max_k) nq = nk = 0;
}

// q is the raw tensor map.q describes (the one-tile 256-column forward reads its rows).
cudaError_t launch_fwd(const Maps& m, const Shape& s, const void* q, void* o, float* lse,
                       cudaStream_t st);
cudaError_t launch_delta(const Shape& s, const void* o, const void* dO, float* delta,
                         cudaStream_t st);
// q and dO are the raw [B*H, N, d] tensors the maps describe (the dQ kernel reads its
// query rows of both directly).
cudaError_t launch_dq(const Maps& m, const Shape& s, const void* q, const void* dO,
                      const float* lse, const float* delta, void* dq, cudaStream_t st);
// k and v are the raw tensors map.k / map.v describe (the d = 64 kernel reads its key rows
// directly into tensor memory).
cudaError_t launch_dkv(const Maps& m, const Shape& s, const void* q, const void* k,
                       const void* v, const void* dO,
                       const float* lse, const float* delta, void* dk, void* dv,
                       cudaStream_t st);

// Split-KV decode: one query row per (b, h) against Nk keys, in `splits` key ranges.
struct DecodeShape {
  int BH, Nk, d, splits;
  bool bf16;
  float scale;
  unsigned long long wait_limit;
  int stall = 0;
};
// Resident CTAs of the decode partial kernel per SM (its shared-memory footprint).
constexpr int kDecodeCtasPerSmPublic = 3;
// Keys per split: ceil(Nk / splits) rounded up to a multiple of 64.
int decode_chunk(int Nk, int splits);
cudaError_t launch_decode_partial(const DecodeShape& s, const void* q, const void* k,
                                  const void* v, float* partials, cudaStream_t st);
cudaError_t launch_decode_merge(const DecodeShape& s, const float* partials, void* o,
                                float* lse, cudaStream_t st);

// Each kernel translation unit has its own device status word; these read (after the
// work queued on `st`, blocking) and clear it. Return the word (0 = no timeout).
int status_fwd(cudaStream_t st, cudaError_t* err);
int status_delta(cudaStream_t st, cudaError_t* err);
int status_dq(cudaStream_t st, cudaError_t* err);
int status_dkv(cudaStream_t st, cudaError_t* err);
int status_decode(cudaStream_t st, cudaError_t* err);

}  // namespace attn

// Defines the status reader of one translation unit.
#define ATTN_DEFINE_STATUS_READER(fn)                                                      \
  int fn(cudaStream_t st, cudaError_t* err) {                                             \
    int h = 0;                                                                             \
    const int zero = 0;                                                                    \
    cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_kernel_status, sizeof(int), 0,        \
                                              cudaMemcpyDeviceToHost, st);                 \
    if (e == cudaSuccess)                                                                  \
      e = cudaMemcpyToSymbolAsync(g_kernel_status, &zero, sizeof(int), 0,                 \
                                  cudaMemcpyHostToDevice, st);                             \
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);                                   \
    *err = e;                                                                              \
    return h;                                                                              \
  }
