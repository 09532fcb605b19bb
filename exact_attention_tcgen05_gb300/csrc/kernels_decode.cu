// kernels_decode.cu - instantiation and launch of the split-KV decode kernels.
#include "decode.cuh"
#include "launch.h"

namespace attn {

static_assert(kDecodeCtasPerSm == kDecodeCtasPerSmPublic, "one value for the split heuristic");
static_assert(3 * (DecodeCfg<128>::kSmemBytes + 1024) <= 228 * 1024, "three CTAs per SM");
static_assert(3 * (DecodeCfg<64>::kSmemBytes + 1024) <= 228 * 1024, "three CTAs per SM");
static_assert(3 * (DecodeCfg<256>::kSmemBytes + 1024) <= 228 * 1024, "three CTAs per SM");

int decode_chunk(int Nk, int splits) {
  const int per = (Nk + splits - 1) / splits;
  return kDecodeSub * ((per + kDecodeSub - 1) / kDecodeSub);
}

template <int D, bool BF16>
static cudaError_t launch_decode_partial_t(const DecodeShape& s, const void* q, const void* k,
                                           const void* v, float* partials, cudaStream_t st) {
  using C = DecodeCfg<D>;
  auto kern = attn_decode_partial_kernel<D, BF16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  DecodeParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.partials = partials;
  p.Nk = s.Nk;
  p.splits = s.splits;
  p.chunk = decode_chunk(s.Nk, s.splits);
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  p.stall = s.stall;
  dim3 grid(s.splits, s.BH);
  kern<<<grid, kDecodeThreads, C::kSmemBytes, st>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_decode_merge_t(const DecodeShape& s, const float* partials, void* o,
                                         float* lse, cudaStream_t st) {
  dim3 grid((s.BH + 7) / 8);
  attn_decode_merge_kernel<D, BF16><<<grid, 256, 0, st>>>(partials, o, lse, s.BH, s.splits);
  return cudaGetLastError();
}

cudaError_t launch_decode_partial(const DecodeShape& s, const void* q, const void* k,
                                  const void* v, float* partials, cudaStream_t st) {
  if (s.d == 256) return s.bf16 ? launch_decode_partial_t<256, true>(s, q, k, v, partials, st)
                                : launch_decode_partial_t<256, false>(s, q, k, v, partials, st);
  if (s.d == 128) return s.bf16 ? launch_decode_partial_t<128, true>(s, q, k, v, partials, st)
                                : launch_decode_partial_t<128, false>(s, q, k, v, partials, st);
  return s.bf16 ? launch_decode_partial_t<64, true>(s, q, k, v, partials, st)
                : launch_decode_partial_t<64, false>(s, q, k, v, partials, st);
}

cudaError_t launch_decode_merge(const DecodeShape& s, const float* partials, void* o,
                                float* lse, cudaStream_t st) {
  if (s.d == 256) return s.bf16 ? launch_decode_merge_t<256, true>(s, partials, o, lse, st)
                                : launch_decode_merge_t<256, false>(s, partials, o, lse, st);
  if (s.d == 128) return s.bf16 ? launch_decode_merge_t<128, true>(s, partials, o, lse, st)
                                : launch_decode_merge_t<128, false>(s, partials, o, lse, st);
  return s.bf16 ? launch_decode_merge_t<64, true>(s, partials, o, lse, st)
                : launch_decode_merge_t<64, false>(s, partials, o, lse, st);
}

ATTN_DEFINE_STATUS_READER(status_decode)

}  // namespace attn
