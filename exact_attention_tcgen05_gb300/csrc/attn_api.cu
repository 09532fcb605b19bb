// attn_api.cu - the C ABI declared in include/attn.h: argument validation (host only,
// before any CUDA call), TMA descriptor encoding and kernel launches on the caller's
// stream. The library allocates no device memory and keeps no per-call state.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <initializer_list>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.h"
#include "launch.h"

namespace {

using attn::Maps;
using attn::Shape;

constexpr int kMaxN = 1 << 20;
constexpr long long kMaxBH = 65535;  // grid.y limit

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;
};
Range range_of(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// Head dimensions the attention kernels take: multiples of 8 (16-byte rows for TMA) up to
// 256; d <= 64 runs on the 64-column kernels, d <= 128 on the 128-column ones, d > 128 on
// the 256-column ones, with the columns past d read as zero. (Split-KV decoding takes
// exactly 64, 128 or 256.)
constexpr int kMaxD = 256;
bool head_dim_ok(int d, int max_d = kMaxD) { return d >= 8 && d <= max_d && d % 8 == 0; }

attn_status check_shape(int B, int H, int N, int d, attn_dtype dtype, int max_d = kMaxD) {
  if (B < 1 || H < 1 || N < 1 || N > kMaxN) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * H > kMaxBH) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(d, max_d)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

attn_status check_scale(float scale) {
  return (std::isfinite(scale) && scale > 0.f) ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

unsigned long long wait_limit_cycles() {
  static const unsigned long long v = [] {
    const char* e = std::getenv("ATTN_WAIT_LIMIT_CYCLES");
    if (e != nullptr) {
      char* end = nullptr;
      const unsigned long long x = std::strtoull(e, &end, 10);
      if (end != e && x > 0) return x;
    }
    return 1ull << 31;  // about one second at the GB300's maximum SM clock
  }();
  return v;
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no link against libcuda).
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// A 3-D 16-bit tiled map with 128-byte swizzle and zero fill. cuTensorMapEncodeTiled is a
// driver call and needs a current context in the calling thread; a thread that has made no
// runtime call yet (an autograd worker thread, say) has none and gets
// CUDA_ERROR_INVALID_CONTEXT. The thread is then bound to its current device's primary
// context (what the runtime's own calls would do) and the encoding retried once.
attn_status encode_3d(CUtensorMap* m, const void* base, bool bf16, const cuuint64_t (&dims)[3],
                      const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3],
                      bool swizzle = true) {
  EncodeFn enc = get_encode();
  if (enc == nullptr) return ATTN_ERR_CUDA;
  const cuuint32_t estr[3] = {1, 1, 1};
  auto encode = [&] {
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
               const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  CUresult r = encode();
  if (r == CUDA_ERROR_INVALID_CONTEXT) {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess) r = encode();
  }
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// [BH, N, d] 16-bit tensor, read as [64-column x 128-row] boxes with 128-byte swizzle;
// rows past N read as zero.
attn_status encode_map(CUtensorMap* m, const void* base, int BH, int N, int d, bool bf16,
                       int box_rows = 128) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * (cuuint64_t)d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  return encode_3d(m, base, bf16, dims, strides, box);
}

// [BH, N, d] 16-bit tensor as a TMA store target in unswizzled [32-column x 32-row] boxes
// (64-byte rows in shared memory).
attn_status encode_map_half_rows(CUtensorMap* m, const void* base, int BH, int N, int d,
                                 bool bf16) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * (cuuint64_t)d * 2};
  const cuuint32_t box[3] = {32, 32, 1};
  return encode_3d(m, base, bf16, dims, strides, box, false);
}

// [total, H, d] packed 16-bit tensor, read as [64-column x 1-head x 128-token] boxes with
// 128-byte swizzle: the same shared-memory image as a [64 x 128] box of the dense map.
// Tokens past `total` read as zero.
attn_status encode_map_packed(CUtensorMap* m, const void* base, int H, int total, int d,
                              bool bf16, int box_rows = 128) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)total};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * (cuuint64_t)d * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  return encode_3d(m, base, bf16, dims, strides, box);
}

// ATTN_TEST_STALL = 1: every kernel's copies are withheld, so that its pipeline waits run
// out (after ATTN_WAIT_LIMIT_CYCLES) on phases that never complete - the failure tests'
// way to exercise the bounded waits and the abort paths without a fault.
int test_stall() {
  static const int v = [] {
    const char* e = std::getenv("ATTN_TEST_STALL");
    return (e != nullptr && e[0] == '1') ? 1 : 0;
  }();
  return v;
}

Shape make_shape(int B, int H, int N, int d, attn_dtype dtype, int causal, float scale,
                 int Nk = -1) {
  Shape s;
  s.BH = B * H;
  s.N = N;
  s.Nk = Nk < 0 ? N : Nk;
  s.d = d;
  s.bf16 = dtype == ATTN_BF16;
  s.causal = causal != 0;
  s.scale = scale;
  s.wait_limit = wait_limit_cycles();
  s.stall = test_stall();
  s.vl = attn::Varlen{};  // dense tensors
  return s;
}

attn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace

extern "C" {

const char* attn_status_str(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
  }
  return "ATTN_ERR_UNKNOWN";
}

size_t attn_bwd_workspace_bytes(int B, int H, int N) {
  if (B <= 0 || H <= 0 || N <= 0) return 0;
  return (size_t)4 * (size_t)B * (size_t)H * (size_t)N;
}

attn_status attn_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int H, int Nq, int Nk, int d, attn_dtype dtype, int causal,
                        float scale, void* cuda_stream) {
  attn_status st = check_shape(B, H, Nq, d, dtype);
  if (st != ATTN_OK) return st;
  if ((st = check_shape(B, H, Nk, d, dtype)) != ATTN_OK) return st;
  if (causal && Nk < Nq) return ATTN_ERR_INVALID_ARG;  // rows would see no key
  if ((st = check_scale(scale)) != ATTN_OK) return st;
  const void* ptrs[5] = {q, k, v, o, lse};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID_ARG;
  const size_t qb = (size_t)B * H * Nq * d * 2, kb = (size_t)B * H * Nk * d * 2;
  const size_t lb = (size_t)B * H * Nq * 4;
  const Range rq = range_of(q, qb), rk = range_of(k, kb), rv = range_of(v, kb);
  const Range ro = range_of(o, qb), rl = range_of(lse, lb);
  for (Range out : {ro, rl})
    for (Range in : {rq, rk, rv})
      if (overlap(out, in)) return ATTN_ERR_INVALID_ARG;
  if (overlap(ro, rl)) return ATTN_ERR_INVALID_ARG;

  const Shape s = make_shape(B, H, Nq, d, dtype, causal, scale, Nk);
  Maps m;
  if ((st = encode_map(&m.q, q, s.BH, Nq, d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map(&m.k, k, s.BH, Nk, d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map(&m.v, v, s.BH, Nk, d, s.bf16)) != ATTN_OK) return st;
  m.d_o = m.v;
  m.k64 = m.k;
  if (d > 64 && (st = encode_map(&m.k64, k, s.BH, Nk, d, s.bf16, 64)) != ATTN_OK) return st;
  m.v64 = m.v;
  if (d > 128 && (st = encode_map(&m.v64, v, s.BH, Nk, d, s.bf16, 64)) != ATTN_OK) return st;
  m.o = m.q;
  if (d <= 64 && (st = encode_map(&m.o, o, s.BH, Nq, d, s.bf16, 32)) != ATTN_OK) return st;
  return from_cuda(attn::launch_fwd(m, s, q, o, lse, static_cast<cudaStream_t>(cuda_stream)));
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, attn_dtype dtype, int causal, float scale,
                     void* cuda_stream) {
  return attn_fwd_qk(q, k, v, o, lse, B, H, N, N, d, dtype, causal, scale, cuda_stream);
}

attn_status attn_bwd_preprocess(const void* o, const void* dO, float* delta, int B, int H,
                                int N, int d, attn_dtype dtype, void* cuda_stream) {
  attn_status st = check_shape(B, H, N, d, dtype);
  if (st != ATTN_OK) return st;
  const void* ptrs[3] = {o, dO, delta};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID_ARG;
  const size_t tb = (size_t)B * H * N * d * 2;
  const Range rd = range_of(delta, (size_t)B * H * N * 4);
  if (overlap(rd, range_of(o, tb)) || overlap(rd, range_of(dO, tb))) return ATTN_ERR_INVALID_ARG;
  const Shape s = make_shape(B, H, N, d, dtype, 0, 1.f);
  return from_cuda(attn::launch_delta(s, o, dO, delta, static_cast<cudaStream_t>(cuda_stream)));
}

namespace {

// Validation shared by the backward entry points. `outs` must not overlap `ins` or
// each other.
attn_status check_ranges(const Range* ins, int n_in, const Range* outs, int n_out) {
  for (int a = 0; a < n_out; ++a) {
    for (int i = 0; i < n_in; ++i)
      if (overlap(outs[a], ins[i])) return ATTN_ERR_INVALID_ARG;
    for (int b = a + 1; b < n_out; ++b)
      if (overlap(outs[a], outs[b])) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

attn_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status encode_bwd_maps(Maps* m, const void* q, const void* k, const void* v,
                            const void* dO, const Shape& s) {
  attn_status st;
  if ((st = encode_map(&m->q, q, s.BH, s.N, s.d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map(&m->k, k, s.BH, s.Nk, s.d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map(&m->v, v, s.BH, s.Nk, s.d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map(&m->d_o, dO, s.BH, s.N, s.d, s.bf16)) != ATTN_OK) return st;
  m->k64 = m->k;
  m->v64 = m->v;
  m->q64 = m->q;
  m->do64 = m->d_o;
  if (s.d <= 128) return ATTN_OK;
  // head dims above 128: the streamed 64-row blocks of the 256-column backward
  if ((st = encode_map(&m->k64, k, s.BH, s.Nk, s.d, s.bf16, 64)) != ATTN_OK) return st;
  if ((st = encode_map(&m->v64, v, s.BH, s.Nk, s.d, s.bf16, 64)) != ATTN_OK) return st;
  if ((st = encode_map(&m->q64, q, s.BH, s.N, s.d, s.bf16, 64)) != ATTN_OK) return st;
  return encode_map(&m->do64, dO, s.BH, s.N, s.d, s.bf16, 64);
}

// The dQ output as a TMA store target (dense, d <= 64: the persistent kernel's staged
// epilogue); otherwise unused and left as a copy of the q map.
attn_status encode_dq_out_map(Maps* m, void* dq, const Shape& s) {
  m->dq = m->q;
  if (s.vl.cu_q != nullptr || s.d > 64) return ATTN_OK;
  return encode_map_half_rows(&m->dq, dq, s.BH, s.N, s.d, s.bf16);
}

// The dK/dV outputs as TMA store targets (dense, d <= 64: the persistent kernel's staged
// epilogue); otherwise unused and left as copies of the input maps.
attn_status encode_dkv_out_maps(Maps* m, void* dk, void* dv, const Shape& s) {
  m->dk = m->dv = m->k;
  if (s.vl.cu_q != nullptr || s.d > 64) return ATTN_OK;
  attn_status st = encode_map(&m->dk, dk, s.BH, s.Nk, s.d, s.bf16, 32);
  if (st == ATTN_OK) st = encode_map(&m->dv, dv, s.BH, s.Nk, s.d, s.bf16, 32);
  return st;
}

}  // namespace

attn_status attn_bwd_dkv(const void* q, const void* k, const void* v, const float* lse,
                         const float* delta, const void* dO, void* dk, void* dv, int B, int H,
                         int N, int d, attn_dtype dtype, int causal, float scale,
                         void* cuda_stream) {
  attn_status st = check_shape(B, H, N, d, dtype);
  if (st != ATTN_OK) return st;
  if ((st = check_scale(scale)) != ATTN_OK) return st;
  if ((st = check_ptrs({q, k, v, lse, delta, dO, dk, dv})) != ATTN_OK) return st;
  const size_t tb = (size_t)B * H * N * d * 2, lb = (size_t)B * H * N * 4;
  const Range ins[6] = {range_of(q, tb),   range_of(k, tb),     range_of(v, tb),
                        range_of(lse, lb), range_of(delta, lb), range_of(dO, tb)};
  const Range outs[2] = {range_of(dk, tb), range_of(dv, tb)};
  if ((st = check_ranges(ins, 6, outs, 2)) != ATTN_OK) return st;
  const Shape s = make_shape(B, H, N, d, dtype, causal, scale);
  Maps m;
  if ((st = encode_bwd_maps(&m, q, k, v, dO, s)) != ATTN_OK) return st;
  if ((st = encode_dkv_out_maps(&m, dk, dv, s)) != ATTN_OK) return st;
  return from_cuda(attn::launch_dkv(m, s, q, k, v, dO, lse, delta, dk, dv,
                                    static_cast<cudaStream_t>(cuda_stream)));
}

attn_status attn_bwd_dq(const void* q, const void* k, const void* v, const float* lse,
                        const float* delta, const void* dO, void* dq, int B, int H, int N,
                        int d, attn_dtype dtype, int causal, float scale, void* cuda_stream) {
  attn_status st = check_shape(B, H, N, d, dtype);
  if (st != ATTN_OK) return st;
  if ((st = check_scale(scale)) != ATTN_OK) return st;
  if ((st = check_ptrs({q, k, v, lse, delta, dO, dq})) != ATTN_OK) return st;
  const size_t tb = (size_t)B * H * N * d * 2, lb = (size_t)B * H * N * 4;
  const Range ins[6] = {range_of(q, tb),   range_of(k, tb),     range_of(v, tb),
                        range_of(lse, lb), range_of(delta, lb), range_of(dO, tb)};
  const Range outs[1] = {range_of(dq, tb)};
  if ((st = check_ranges(ins, 6, outs, 1)) != ATTN_OK) return st;
  const Shape s = make_shape(B, H, N, d, dtype, causal, scale);
  Maps m;
  if ((st = encode_bwd_maps(&m, q, k, v, dO, s)) != ATTN_OK) return st;
  if ((st = encode_dq_out_map(&m, dq, s)) != ATTN_OK) return st;
  return from_cuda(
      attn::launch_dq(m, s, q, dO, lse, delta, dq, static_cast<cudaStream_t>(cuda_stream)));
}

attn_status attn_bwd_qk(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dO, void* dq, void* dk, void* dv,
                        void* workspace, int B, int H, int Nq, int Nk, int d,
                        attn_dtype dtype, int causal, float scale, void* cuda_stream) {
  attn_status st = check_shape(B, H, Nq, d, dtype);
  if (st != ATTN_OK) return st;
  if ((st = check_shape(B, H, Nk, d, dtype)) != ATTN_OK) return st;
  if (causal && Nk < Nq) return ATTN_ERR_INVALID_ARG;
  if ((st = check_scale(scale)) != ATTN_OK) return st;
  if ((st = check_ptrs({q, k, v, o, lse, dO, dq, dk, dv, workspace})) != ATTN_OK) return st;
  const size_t qb = (size_t)B * H * Nq * d * 2, kb = (size_t)B * H * Nk * d * 2;
  const size_t lb = (size_t)B * H * Nq * 4;
  const Range ins[6] = {range_of(q, qb), range_of(k, kb),   range_of(v, kb),
                        range_of(o, qb), range_of(lse, lb), range_of(dO, qb)};
  const Range outs[4] = {range_of(dq, qb), range_of(dk, kb), range_of(dv, kb),
                         range_of(workspace, lb)};
  if ((st = check_ranges(ins, 6, outs, 4)) != ATTN_OK) return st;

  const Shape s = make_shape(B, H, Nq, d, dtype, causal, scale, Nk);
  Maps m;
  if ((st = encode_bwd_maps(&m, q, k, v, dO, s)) != ATTN_OK) return st;
  if ((st = encode_dkv_out_maps(&m, dk, dv, s)) != ATTN_OK) return st;
  if ((st = encode_dq_out_map(&m, dq, s)) != ATTN_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(cuda_stream);
  float* delta = static_cast<float*>(workspace);
  cudaError_t e = attn::launch_delta(s, o, dO, delta, cs);
  if (e == cudaSuccess) e = attn::launch_dkv(m, s, q, k, v, dO, lse, delta, dk, dv, cs);
  if (e == cudaSuccess) e = attn::launch_dq(m, s, q, dO, lse, delta, dq, cs);
  return from_cuda(e);
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, void* dq, void* dk, void* dv,
                     void* workspace, int B, int H, int N, int d, attn_dtype dtype, int causal,
                     float scale, void* cuda_stream) {
  return attn_bwd_qk(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, H, N, N, d, dtype, causal,
                     scale, cuda_stream);
}

// ---------------------------------------------------------------- packed batches
namespace {

// Sizes of a packed variable-length call; the per-sequence bounds in cu_seqlens live in
// device memory and are checked by the kernels.
attn_status check_varlen(int B, int H, int total_q, int total_k, int max_q, int max_k, int d,
                         attn_dtype dtype, const int* cu_q, const int* cu_k) {
  if (B < 1 || H < 1 || (long long)B * H > kMaxBH) return ATTN_ERR_INVALID_ARG;
  if (total_q < 1 || total_k < 1) return ATTN_ERR_INVALID_ARG;
  if (max_q < 1 || max_q > kMaxN || max_q > total_q) return ATTN_ERR_INVALID_ARG;
  if (max_k < 1 || max_k > kMaxN || max_k > total_k) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (cu_q == nullptr || cu_k == nullptr) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cu_q) | reinterpret_cast<uintptr_t>(cu_k)) & 3u)
    return ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(d)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

Shape make_varlen_shape(int B, int H, int total_q, int total_k, int max_q, int max_k, int d,
                        attn_dtype dtype, int causal, float scale, const int* cu_q,
                        const int* cu_k, const int* host_cu_q, const int* host_cu_k) {
  Shape s = make_shape(B, H, max_q, d, dtype, causal, scale, max_k);
  s.host_cu_q = host_cu_q;
  s.host_cu_k = host_cu_k;
  s.vl_b = B;
  s.vl.cu_q = cu_q;
  s.vl.cu_k = cu_k;
  s.vl.H = H;
  s.vl.total_q = total_q;
  s.vl.total_k = total_k;
  s.vl.max_q = max_q;
  s.vl.max_k = max_k;
  return s;
}

}  // namespace

size_t attn_bwd_varlen_workspace_bytes(int H, int total_q) {
  if (H <= 0 || total_q <= 0) return 0;
  return (size_t)4 * (size_t)H * (size_t)total_q;
}

attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens_q, const int* cu_seqlens_k,
                            const int* cu_seqlens_q_host, const int* cu_seqlens_k_host, int B,
                            int H, int total_q, int total_k, int max_seqlen_q,
                            int max_seqlen_k, int d, attn_dtype dtype, int causal, float scale,
                            void* cuda_stream) {
  attn_status st = check_varlen(B, H, total_q, total_k, max_seqlen_q, max_seqlen_k, d, dtype,
                                cu_seqlens_q, cu_seqlens_k);
  if (st != ATTN_OK) return st;
  if ((cu_seqlens_q_host == nullptr) != (cu_seqlens_k_host == nullptr))
    return ATTN_ERR_INVALID_ARG;
  if ((st = check_scale(scale)) != ATTN_OK) return st;
  if ((st = check_ptrs({q, k, v, o, lse})) != ATTN_OK) return st;
  const size_t qb = (size_t)total_q * H * d * 2, kb = (size_t)total_k * H * d * 2;
  const size_t lb = (size_t)H * total_q * 4;
  const Range ins[5] = {range_of(q, qb), range_of(k, kb), range_of(v, kb),
                        range_of(cu_seqlens_q, (size_t)(B + 1) * 4),
                        range_of(cu_seqlens_k, (size_t)(B + 1) * 4)};
  const Range outs[2] = {range_of(o, qb), range_of(lse, lb)};
  if ((st = check_ranges(ins, 5, outs, 2)) != ATTN_OK) return st;

  const Shape s = make_varlen_shape(B, H, total_q, total_k, max_seqlen_q, max_seqlen_k, d,
                                    dtype, causal, scale, cu_seqlens_q, cu_seqlens_k,
                                    cu_seqlens_q_host, cu_seqlens_k_host);
  Maps m;
  if ((st = encode_map_packed(&m.q, q, H, total_q, d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map_packed(&m.k, k, H, total_k, d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map_packed(&m.v, v, H, total_k, d, s.bf16)) != ATTN_OK) return st;
  m.d_o = m.v;
  m.k64 = m.k;
  if (d > 64 && (st = encode_map_packed(&m.k64, k, H, total_k, d, s.bf16, 64)) != ATTN_OK)
    return st;
  m.v64 = m.v;
  if (d > 128 && (st = encode_map_packed(&m.v64, v, H, total_k, d, s.bf16, 64)) != ATTN_OK)
    return st;
  m.o = m.q;  // packed batches keep the row stores
  return from_cuda(attn::launch_fwd(m, s, q, o, lse, static_cast<cudaStream_t>(cuda_stream)));
}

attn_status attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dO, void* dq, void* dk, void* dv,
                            void* workspace, const int* cu_seqlens_q, const int* cu_seqlens_k,
                            const int* cu_seqlens_q_host, const int* cu_seqlens_k_host, int B,
                            int H, int total_q, int total_k, int max_seqlen_q,
                            int max_seqlen_k, int d, attn_dtype dtype, int causal, float scale,
                            void* cuda_stream) {
  attn_status st = check_varlen(B, H, total_q, total_k, max_seqlen_q, max_seqlen_k, d, dtype,
                                cu_seqlens_q, cu_seqlens_k);
  if (st == ATTN_OK && (cu_seqlens_q_host == nullptr) != (cu_seqlens_k_host == nullptr))
    st = ATTN_ERR_INVALID_ARG;
  if (st != ATTN_OK) return st;
  if ((st = check_scale(scale)) != ATTN_OK) return st;
  if ((st = check_ptrs({q, k, v, o, lse, dO, dq, dk, dv, workspace})) != ATTN_OK) return st;
  const size_t qb = (size_t)total_q * H * d * 2, kb = (size_t)total_k * H * d * 2;
  const size_t lb = (size_t)H * total_q * 4;
  const Range ins[8] = {range_of(q, qb), range_of(k, kb),   range_of(v, kb),
                        range_of(o, qb), range_of(lse, lb), range_of(dO, qb),
                        range_of(cu_seqlens_q, (size_t)(B + 1) * 4),
                        range_of(cu_seqlens_k, (size_t)(B + 1) * 4)};
  const Range outs[4] = {range_of(dq, qb), range_of(dk, kb), range_of(dv, kb),
                         range_of(workspace, lb)};
  if ((st = check_ranges(ins, 8, outs, 4)) != ATTN_OK) return st;

  const Shape s = make_varlen_shape(B, H, total_q, total_k, max_seqlen_q, max_seqlen_k, d,
                                    dtype, causal, scale, cu_seqlens_q, cu_seqlens_k,
                                    cu_seqlens_q_host, cu_seqlens_k_host);
  Maps m;
  if ((st = encode_map_packed(&m.q, q, H, total_q, d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map_packed(&m.k, k, H, total_k, d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map_packed(&m.v, v, H, total_k, d, s.bf16)) != ATTN_OK) return st;
  if ((st = encode_map_packed(&m.d_o, dO, H, total_q, d, s.bf16)) != ATTN_OK) return st;
  m.k64 = m.k;
  m.v64 = m.v;
  m.q64 = m.q;
  m.do64 = m.d_o;
  if (d > 128) {  // the streamed 64-row blocks of the 256-column backward
    if ((st = encode_map_packed(&m.k64, k, H, total_k, d, s.bf16, 64)) != ATTN_OK) return st;
    if ((st = encode_map_packed(&m.v64, v, H, total_k, d, s.bf16, 64)) != ATTN_OK) return st;
    if ((st = encode_map_packed(&m.q64, q, H, total_q, d, s.bf16, 64)) != ATTN_OK) return st;
    if ((st = encode_map_packed(&m.do64, dO, H, total_q, d, s.bf16, 64)) != ATTN_OK) return st;
  }
  if ((st = encode_dkv_out_maps(&m, dk, dv, s)) != ATTN_OK) return st;  // unused: packed
  if ((st = encode_dq_out_map(&m, dq, s)) != ATTN_OK) return st;        // unused: packed
  cudaStream_t cs = static_cast<cudaStream_t>(cuda_stream);
  float* delta = static_cast<float*>(workspace);
  cudaError_t e = attn::launch_delta(s, o, dO, delta, cs);
  if (e == cudaSuccess) e = attn::launch_dkv(m, s, q, k, v, dO, lse, delta, dk, dv, cs);
  if (e == cudaSuccess) e = attn::launch_dq(m, s, q, dO, lse, delta, dq, cs);
  return from_cuda(e);
}

// ---------------------------------------------------------------- host-buffer step
namespace {
// Chunk boundaries of the host-buffer step: `chunks` chunks of B*H slices whose sizes ramp up
// and down (weights 1, 2, 3, 3, ..., 3, 2, 1), so that the first upload, which nothing
// overlaps, and the last chunk's compute and download, which nothing overlaps either, are
// short. bounds[c] .. bounds[c+1] are the slices of chunk c. Returns the largest chunk.
long long step_schedule(long long bh, int chunks, std::vector<long long>& bounds) {
  std::vector<long long> w(chunks);
  long long wsum = 0;
  for (int c = 0; c < chunks; ++c) {
    w[c] = std::min<long long>({(long long)c + 1, (long long)chunks - c, 3});
    wsum += w[c];
  }
  bounds.assign(chunks + 1, 0);
  long long acc = 0, largest = 0;
  for (int c = 0; c < chunks; ++c) {
    acc += w[c];
    // at least one slice per chunk, and room for one per remaining chunk
    long long b = std::max<long long>(bounds[c] + 1, (bh * acc + wsum / 2) / wsum);
    b = std::min<long long>(b, bh - (chunks - 1 - c));
    bounds[c + 1] = b;
    largest = std::max(largest, b - bounds[c]);
  }
  return largest;
}
// Device buffer sets used in turn: chunk c's inputs go into set c % kStepSets once chunk
// c - kStepSets has been computed, and its outputs once chunk c - kStepSets's outputs have
// been copied out. (A third set measured no faster on GB300: the host link bounds the step.)
constexpr int kStepSets = 2;
size_t step_set_bytes(long long slices, int N, int d) {
  const size_t t = (size_t)slices * N * d * 2, r = (size_t)slices * N * 4;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return 8 * up(t) + 2 * up(r);
}
}  // namespace

namespace {
// attn_step_host's two side streams and kNumEv x chunks events, per CUDA context (streams and
// events belong to the context current when they are made), created on the first call in
// that context and kept until the process exits: creating and destroying them on every
// call costs time inside the step.
// Per chunk: Q/K/V in, dO in, forward done, dK/dV done, all compute done, O/L out,
// dK/dV out, dQ out.
enum StepEvent { kEvQKV, kEvDO, kEvFwd, kEvDKV, kEvComp, kEvOutO, kEvOutKV, kEvOut, kNumEv };
struct StepResources {
  CUcontext ctx = nullptr;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr;
  std::vector<cudaEvent_t> ev[kNumEv];
};
std::mutex g_step_mu;
std::vector<StepResources*> g_step_res;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return nullptr;
  }();
  return fn;
}

cudaError_t new_event(cudaEvent_t* ev) {
  return cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
}

// The resources of the calling thread's current context with at least `chunks` events of
// each kind (call with g_step_mu held). A thread without a current context is bound to its
// device's primary context by the first runtime call, as any runtime call would.
cudaError_t step_resources(int chunks, StepResources** out) {
  CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx == nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  StepResources* r = nullptr;
  for (StepResources* x : g_step_res)
    if (x->ctx == ctx) r = x;
  if (r == nullptr) {
    r = new StepResources;
    r->ctx = ctx;
    cudaError_t e = cudaStreamCreateWithFlags(&r->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&r->s_out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = new_event(&r->start);
    if (e != cudaSuccess) {
      if (r->s_in) cudaStreamDestroy(r->s_in);
      if (r->s_out) cudaStreamDestroy(r->s_out);
      delete r;
      return e;
    }
    g_step_res.push_back(r);
  }
  while ((int)r->ev[0].size() < chunks) {
    cudaEvent_t x[kNumEv] = {};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < kNumEv && e == cudaSuccess; ++i) e = new_event(&x[i]);
    if (e != cudaSuccess) {
      for (cudaEvent_t y : x)
        if (y) cudaEventDestroy(y);
      return e;
    }
    for (int i = 0; i < kNumEv; ++i) r->ev[i].push_back(x[i]);
  }
  *out = r;
  return cudaSuccess;
}
}  // namespace

size_t attn_step_host_scratch_bytes(int B, int H, int N, int d, int chunks) {
  if (B <= 0 || H <= 0 || N <= 0 || chunks <= 0 || !head_dim_ok(d)) return 0;
  const long long bh = (long long)B * H;
  const int c = (int)std::min<long long>(chunks, bh);
  std::vector<long long> bounds;
  return kStepSets * step_set_bytes(step_schedule(bh, c, bounds), N, d);
}

attn_status attn_step_host(const void* q, const void* k, const void* v, const void* dO,
                           void* o, float* lse, void* dq, void* dk, void* dv, void* scratch,
                           size_t scratch_bytes, int B, int H, int N, int d, attn_dtype dtype,
                           int causal, float scale, int chunks, void* cuda_stream) {
  attn_status st = check_shape(B, H, N, d, dtype);
  if (st != ATTN_OK) return st;
  if ((st = check_scale(scale)) != ATTN_OK) return st;
  if (chunks < 1) return ATTN_ERR_INVALID_ARG;
  const void* ptrs[10] = {q, k, v, dO, o, lse, dq, dk, dv, scratch};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  chunks = (int)std::min<long long>(chunks, bh);
  if (scratch_bytes < attn_step_host_scratch_bytes(B, H, N, d, chunks))
    return ATTN_ERR_INVALID_ARG;
  std::vector<long long> bounds;
  const long long per = step_schedule(bh, chunks, bounds);  // the largest chunk
  const size_t row_t = (size_t)N * d * 2, row_r = (size_t)N * 4;  // bytes per slice
  const size_t set_bytes = step_set_bytes(per, N, d);
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };

  cudaStream_t cs = static_cast<cudaStream_t>(cuda_stream);
  // The side streams and events of this context, created on its first call and kept; the
  // lock is held while this call enqueues its work, so concurrent calls never re-record
  // an event another call is still queueing waits on (waits already queued keep the
  // state the event had when they were queued).
  std::lock_guard<std::mutex> lock(g_step_mu);
  StepResources* res = nullptr;
  cudaError_t e = step_resources(chunks, &res);
  if (e != cudaSuccess) return from_cuda(e);
  cudaStream_t s_in = res->s_in, s_out = res->s_out;
  cudaEvent_t start = res->start;
  const std::vector<cudaEvent_t>(&ev)[kNumEv] = res->ev;
  // The side streams start after the work already queued on the caller's stream.
  e = cudaEventRecord(start, cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, start, 0);
  auto rec = [&](StepEvent k, int c, cudaStream_t st_) {
    if (e == cudaSuccess) e = cudaEventRecord(ev[k][c], st_);
  };
  auto wait = [&](cudaStream_t st_, StepEvent k, int c) {  // no wait for c < 0
    if (e == cudaSuccess && c >= 0) e = cudaStreamWaitEvent(st_, ev[k][c], 0);
  };
  auto h2d = [&](void* dst, const void* src, size_t bytes) {
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s_in);
  };
  auto d2h = [&](void* dst, const void* src, size_t bytes) {
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s_out);
  };
  auto run = [&](attn_status x) {
    if (e == cudaSuccess && st == ATTN_OK) st = x;
  };

  // Chunk c uses buffer set c % kStepSets, which chunk p = c - kStepSets used before: each
  // buffer is refilled only once p's last reader of it has run (inputs: p's backward;
  // O/L, dK/dV, dQ: p's copies of them out). Each output leaves as soon as its kernel is
  // done, so that the last chunk's O and dK/dV copies overlap its remaining kernels.
  for (int c = 0; c < chunks && e == cudaSuccess && st == ATTN_OK; ++c) {
    const int p = c - kStepSets;
    const long long b0 = bounds[c];
    const long long n = bounds[c + 1] - b0;
    uint8_t* set = static_cast<uint8_t*>(scratch) + (size_t)(c % kStepSets) * set_bytes;
    uint8_t* dev[8];  // q, k, v, dO, o, dq, dk, dv
    for (int i = 0; i < 8; ++i) dev[i] = set + (size_t)i * up((size_t)per * row_t);
    float* d_lse = reinterpret_cast<float*>(set + 8 * up((size_t)per * row_t));
    float* d_delta = reinterpret_cast<float*>(set + 8 * up((size_t)per * row_t) +
                                              up((size_t)per * row_r));
    const size_t tb = (size_t)n * row_t, rb = (size_t)n * row_r;
    const size_t off_t = (size_t)b0 * row_t, off_r = (size_t)b0 * row_r;
    auto host_at = [&](const void* base) { return static_cast<const uint8_t*>(base) + off_t; };
    auto host_out = [&](void* base, size_t off) { return static_cast<uint8_t*>(base) + off; };
    const int ni = (int)n;
    // inputs: Q, K, V (the forward's), then dO
    wait(s_in, kEvComp, p);
    h2d(dev[0], host_at(q), tb);
    h2d(dev[1], host_at(k), tb);
    h2d(dev[2], host_at(v), tb);
    rec(kEvQKV, c, s_in);
    h2d(dev[3], host_at(dO), tb);
    rec(kEvDO, c, s_in);
    // forward, then the backward's three kernels, on the caller's stream
    wait(cs, kEvQKV, c);
    wait(cs, kEvOutO, p);
    if (e == cudaSuccess)
      run(attn_fwd(dev[0], dev[1], dev[2], dev[4], d_lse, 1, ni, N, d, dtype, causal, scale,
                   cs));
    rec(kEvFwd, c, cs);
    wait(cs, kEvDO, c);
    if (e == cudaSuccess && st == ATTN_OK)
      run(attn_bwd_preprocess(dev[4], dev[3], d_delta, 1, ni, N, d, dtype, cs));
    wait(cs, kEvOutKV, p);
    if (e == cudaSuccess && st == ATTN_OK)
      run(attn_bwd_dkv(dev[0], dev[1], dev[2], d_lse, d_delta, dev[3], dev[6], dev[7], 1, ni,
                       N, d, dtype, causal, scale, cs));
    rec(kEvDKV, c, cs);
    wait(cs, kEvOut, p);
    if (e == cudaSuccess && st == ATTN_OK)
      run(attn_bwd_dq(dev[0], dev[1], dev[2], d_lse, d_delta, dev[3], dev[5], 1, ni, N, d,
                      dtype, causal, scale, cs));
    rec(kEvComp, c, cs);
    // outputs, each after its kernel
    wait(s_out, kEvFwd, c);
    d2h(host_out(o, off_t), dev[4], tb);
    d2h(host_out(lse, off_r), d_lse, rb);
    rec(kEvOutO, c, s_out);
    wait(s_out, kEvDKV, c);
    d2h(host_out(dk, off_t), dev[6], tb);
    d2h(host_out(dv, off_t), dev[7], tb);
    rec(kEvOutKV, c, s_out);
    wait(s_out, kEvComp, c);
    d2h(host_out(dq, off_t), dev[5], tb);
    rec(kEvOut, c, s_out);
  }
  // The caller's stream completes after the last copy out.
  if (st == ATTN_OK) wait(cs, kEvOut, chunks - 1);
  if (st != ATTN_OK) return st;
  return from_cuda(e);
}

// ---------------------------------------------------------------- split-KV decode
namespace {
constexpr int kMaxSplits = 65535;  // grid.x of the partial kernel

attn_status check_decode(int B, int H, int Nk, int d, attn_dtype dtype, int splits) {
  attn_status st = check_shape(B, H, Nk, d, dtype);
  if (st != ATTN_OK) return st;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;  // the kernels' widths
  if (splits < 1 || splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn::DecodeShape make_decode_shape(int B, int H, int Nk, int d, attn_dtype dtype, int splits,
                                    float scale) {
  attn::DecodeShape s;
  s.BH = B * H;
  s.Nk = Nk;
  s.d = d;
  s.splits = splits;
  s.bf16 = dtype == ATTN_BF16;
  s.scale = scale;
  s.wait_limit = wait_limit_cycles();
  s.stall = test_stall();
  return s;
}
}  // namespace

size_t attn_decode_workspace_bytes(int B, int H, int d, int num_splits) {
  if (B <= 0 || H <= 0 || num_splits <= 0 || (d != 64 && d != 128 && d != 256)) return 0;
  return (size_t)4 * (size_t)B * (size_t)H * (size_t)num_splits * (size_t)(d + 4);
}

int attn_decode_splits(int B, int H, int Nk) {
  if (B <= 0 || H <= 0 || Nk <= 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    sms = 152;
  // At least eight waves of resident CTAs, no split shorter than 256 keys, and among the
  // counts up to twice that the one whose last wave is fullest.
  const long long bh = (long long)B * H;
  const long long resident = (long long)sms * attn::kDecodeCtasPerSmPublic;
  const long long most = std::min(std::max(1LL, ((long long)Nk + 255) / 256),
                                  (long long)kMaxSplits);
  const long long lo = std::min(most, std::max(1LL, (8 * resident + bh - 1) / bh));
  long long best = lo;
  double best_fill = 0.0;
  for (long long s = lo; s <= std::min(most, 2 * lo); ++s) {
    const long long ctas = bh * s;
    const long long waves = (ctas + resident - 1) / resident;
    const double fill = (double)ctas / (double)(waves * resident);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = s;
    }
  }
  return (int)best;
}

attn_status attn_decode_partial(const void* q, const void* k, const void* v, float* partials,
                                int B, int H, int Nk, int d, attn_dtype dtype, float scale,
                                int num_splits, void* cuda_stream) {
  attn_status st = check_decode(B, H, Nk, d, dtype, num_splits);
  if (st != ATTN_OK) return st;
  if ((st = check_scale(scale)) != ATTN_OK) return st;
  const void* ptrs[4] = {q, k, v, partials};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID_ARG;
  const size_t qb = (size_t)B * H * d * 2, kb = (size_t)B * H * Nk * d * 2;
  const Range rp = range_of(partials, attn_decode_workspace_bytes(B, H, d, num_splits));
  for (Range in : {range_of(q, qb), range_of(k, kb), range_of(v, kb)})
    if (overlap(rp, in)) return ATTN_ERR_INVALID_ARG;
  const attn::DecodeShape s = make_decode_shape(B, H, Nk, d, dtype, num_splits, scale);
  return from_cuda(
      attn::launch_decode_partial(s, q, k, v, partials, static_cast<cudaStream_t>(cuda_stream)));
}

attn_status attn_decode_merge(const float* partials, void* o, float* lse, int B, int H, int d,
                              attn_dtype dtype, int num_splits, void* cuda_stream) {
  attn_status st = check_decode(B, H, 1, d, dtype, num_splits);
  if (st != ATTN_OK) return st;
  const void* ptrs[3] = {partials, o, lse};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID_ARG;
  const Range rp = range_of(partials, attn_decode_workspace_bytes(B, H, d, num_splits));
  const Range ro = range_of(o, (size_t)B * H * d * 2), rl = range_of(lse, (size_t)B * H * 4);
  if (overlap(rp, ro) || overlap(rp, rl) || overlap(ro, rl)) return ATTN_ERR_INVALID_ARG;
  const attn::DecodeShape s = make_decode_shape(B, H, 1, d, dtype, num_splits, 1.f);
  return from_cuda(
      attn::launch_decode_merge(s, partials, o, lse, static_cast<cudaStream_t>(cuda_stream)));
}

attn_status attn_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                        float* partials, int B, int H, int Nk, int d, attn_dtype dtype,
                        float scale, int num_splits, void* cuda_stream) {
  attn_status st = check_decode(B, H, Nk, d, dtype, num_splits);
  if (st != ATTN_OK) return st;
  if (o == nullptr || lse == nullptr || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  const size_t qb = (size_t)B * H * d * 2, kb = (size_t)B * H * Nk * d * 2;
  const Range ro = range_of(o, qb), rl = range_of(lse, (size_t)B * H * 4);
  for (Range out : {ro, rl})
    for (Range in : {range_of(q, qb), range_of(k, kb), range_of(v, kb)})
      if (overlap(out, in)) return ATTN_ERR_INVALID_ARG;
  if ((st = attn_decode_partial(q, k, v, partials, B, H, Nk, d, dtype, scale, num_splits,
                                cuda_stream)) != ATTN_OK)
    return st;
  return attn_decode_merge(partials, o, lse, B, H, d, dtype, num_splits, cuda_stream);
}

attn_status attn_last_kernel_status(void* cuda_stream, int* where) {
  cudaStream_t cs = static_cast<cudaStream_t>(cuda_stream);
  int first = 0;
  using Reader = int (*)(cudaStream_t, cudaError_t*);
  const Reader readers[5] = {attn::status_fwd, attn::status_delta, attn::status_dq,
                             attn::status_dkv, attn::status_decode};
  for (Reader r : readers) {
    cudaError_t e = cudaSuccess;
    const int w = r(cs, &e);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    if (first == 0 && w != 0) first = w;
  }
  if (where != nullptr) *where = first;
  if (first == attn::kStatusBadSeqlens) return ATTN_ERR_INVALID_ARG;
  // a kernel that found its launch unusable and did nothing (shared memory not aligned,
  // the two tensor-memory allocations of a CTA pair at different addresses)
  if (first == attn::kStatusSmemAlign || first == attn::kStatusPairTmem) return ATTN_ERR_CUDA;
  return first == 0 ? ATTN_OK : ATTN_ERR_TIMEOUT;
}

}  // extern "C"
