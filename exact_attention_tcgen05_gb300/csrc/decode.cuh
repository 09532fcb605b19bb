// decode.cuh - split-KV decoding on sm_103a: one query row per (b, h) against a long
// K/V, the keys split into chunks whose partial results are joined afterwards.
//
// Method ("FlashAttentionを1から — 計算を増やして速くする逆説", section その後の版と、推論
// での事情): with a single query token there are no query rows to spread over the GPU,
// so the K/V side is split, each split computes its partial state in parallel, and the
// three update equations of the online softmax (same page, section オンラインsoftmax:
// 途中経過を、後から縮める) join them into the exact result:
//   m' = max(m, m~),  l' = e^(m - m') l + e^(m~ - m') l~,
//   O~' = e^(m - m') O~ + e^(m~ - m') O~_part,     O = O~ / l,  L = m + ln l.
//
// GB300 design. The work is a matrix-vector product per (b, h): every K and V byte is
// read once and used for one multiply-add, so it is HBM-bound and stays on the CUDA
// cores (no tensor-core reshaping).
//  * Partial kernel: one CTA per (split, b·h), 256 threads. K and V rows of the split
//    arrive in 64-key sub-blocks through a ring of shared-memory stages, each filled by
//    two 1-D bulk copies (cp.async.bulk: the rows of a sub-block are contiguous in HBM),
//    so several tens of KiB per SM are in flight without holding registers. Per
//    sub-block: each warp forms eight scores (a lane multiplies D/32 elements, a
//    butterfly of shuffles sums them), warp 0 updates the running max / sum and writes
//    the exp2 weights, and every thread accumulates two output columns over a half
//    (D = 256), a quarter (D = 128) or an eighth (D = 64) of the sub-block's keys. exp is exp2 with
//    scale·log2(e) folded into the score ("Triton 05: Flash Attention", section
//    2. exp -> exp2 트릭). The record written per split is (O~ [D], m, l) in fp32, m in
//    natural-log units.
//  * Merge kernel: one warp per (b, h) reads its splits' records and applies the three
//    equations in fp32; writes O (16-bit) and L.
#pragma once

#include "common.cuh"

namespace attn {

constexpr int kDecodeSub = 64;        // keys per sub-block; split lengths are multiples
constexpr int kDecodeThreads = 256;
constexpr int kDecodeCtasPerSm = 3;   // resident partial-kernel CTAs per SM (shared memory)

struct DecodeParams {
  const void* q;      // [BH, d]
  const void* k;      // [BH, Nk, d]
  const void* v;
  float* partials;    // [BH, S, d + 4]: O~ [d], m, l, 2 unused
  int Nk;
  int splits;         // S
  int chunk;          // keys per split (multiple of kDecodeSub)
  float scale_log2;   // scale * log2(e)
  unsigned long long wait_limit;
  int stall;          // failure tests: thread 0 withholds every copy
};

template <int D>
struct DecodeCfg {
  // 64 KiB of stages (one sub-block of K and V at d = 256, two at d = 128, four at d = 64):
  // three CTAs fit on an SM, about 190 KiB of copies in flight per SM.
  static constexpr int kStages = 64 * 1024 / (2 * kDecodeSub * D * 2);
  static_assert(kStages >= 1, "one stage at least");
  static constexpr int kSubBytes = kDecodeSub * D * 2;  // one K (or V) sub-block
  static constexpr int kStageBytes = 2 * kSubBytes;     // K then V
  static constexpr int kOffScores = kStages * kStageBytes;           // float[64]
  static constexpr int kOffP = kOffScores + kDecodeSub * 4;          // float[64]
  static constexpr int kOffStat = kOffP + kDecodeSub * 4;            // float[4]
  static constexpr int kOffRed = kOffStat + 16;                      // float[groups][D]
  static constexpr int kGroups = kDecodeThreads / (D / 2);           // key groups
  static constexpr int kOffBar = kOffRed + kGroups * D * 4;
  static constexpr int kSmemBytes = kOffBar + kStages * 8 + 16 + 128;  // + alignment
  static constexpr int kRecord = D + 4;                               // floats per split
};

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kDecodeThreads)
    attn_decode_partial_kernel(const DecodeParams p) {
  using C = DecodeCfg<D>;
  constexpr int NS = C::kStages;
  constexpr int kPerLane = D / 32;  // elements of a key row per lane in the score
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  float* sc = reinterpret_cast<float*>(smem + C::kOffScores);
  float* pw = reinterpret_cast<float*>(smem + C::kOffP);
  float* stat = reinterpret_cast<float*>(smem + C::kOffStat);  // [0] alpha
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + NS * 8);

  const int split = blockIdx.x;
  const int bh = blockIdx.y;
  const int warp = warp_id();
  const int lane = lane_id();
  const int k0 = min(p.Nk, split * p.chunk);
  const int k1 = min(p.Nk, k0 + p.chunk);
  const int nsub = (k1 - k0 + kDecodeSub - 1) / kDecodeSub;
  const uint8_t* kbase = reinterpret_cast<const uint8_t*>(p.k) +
                         ((size_t)bh * p.Nk + k0) * (size_t)(D * 2);
  const uint8_t* vbase = reinterpret_cast<const uint8_t*>(p.v) +
                         ((size_t)bh * p.Nk + k0) * (size_t)(D * 2);
  const uint64_t limit = p.wait_limit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Sub-block i of the split: keys [k0 + 64 i, ...), rows (and bytes) it holds.
  auto rows_of = [&](int i) { return min(kDecodeSub, k1 - k0 - i * kDecodeSub); };
  int issued = 0;  // sub-blocks whose copies thread 0 has started
  auto issue = [&](int i) {
    ++issued;
    const int s = i % NS;
    const uint32_t bytes = (uint32_t)rows_of(i) * (uint32_t)(D * 2);
    uint8_t* st = smem + s * C::kStageBytes;
    mbar_arrive_expect_tx(&full[s], 2 * bytes);
    bulk_load(st, kbase + (size_t)i * C::kSubBytes, bytes, &full[s]);
    bulk_load(st + C::kSubBytes, vbase + (size_t)i * C::kSubBytes, bytes, &full[s]);
  };
  if (threadIdx.x == 0 && !p.stall)  // failure tests: no copies, so the waits run out
    for (int i = 0; i < min(NS, nsub); ++i) issue(i);

  // This lane's slice of q, as floats.
  float qv[kPerLane];
  {
    const uint8_t* qrow = reinterpret_cast<const uint8_t*>(p.q) + (size_t)bh * (D * 2);
    if constexpr (kPerLane == 8) {
      const uint4 raw = *reinterpret_cast<const uint4*>(qrow + lane * 16);
      const float2 a = unpack2<BF16>(raw.x), b = unpack2<BF16>(raw.y);
      const float2 c = unpack2<BF16>(raw.z), e = unpack2<BF16>(raw.w);
      qv[0] = a.x; qv[1] = a.y; qv[2] = b.x; qv[3] = b.y;
      qv[4] = c.x; qv[5] = c.y; qv[6] = e.x; qv[7] = e.y;
    } else if constexpr (kPerLane == 4) {
      const uint2 raw = *reinterpret_cast<const uint2*>(qrow + lane * 8);
      const float2 a = unpack2<BF16>(raw.x), b = unpack2<BF16>(raw.y);
      qv[0] = a.x; qv[1] = a.y; qv[2] = b.x; qv[3] = b.y;
    } else {
      const float2 a = unpack2<BF16>(*reinterpret_cast<const uint32_t*>(qrow + lane * 4));
      qv[0] = a.x; qv[1] = a.y;
    }
  }
  const int cp = threadIdx.x % (D / 2);  // this thread's output column pair
  const int kg = threadIdx.x / (D / 2);  // and key group
  constexpr int kKeysPerGroup = kDecodeSub / C::kGroups;
  float2 acc = make_float2(0.f, 0.f);
  float m_run = -INFINITY;  // running max of scale*log2(e)*s (warp 0 keeps it)
  float l_run = 0.f;        // running sum of exp2 weights (warp 0)
  bool ok = true;

  for (int i = 0; i < nsub; ++i) {
    const int s = i % NS;
    const int nvalid = rows_of(i);
    const uint8_t* kst = smem + s * C::kStageBytes;
    const uint8_t* vst = kst + C::kSubBytes;
    if (ok) ok = mbar_wait(&full[s], (i / NS) & 1, limit, abort_flag, kWaitDecFull);
    // ---- scores of the sub-block: warp w takes keys w, w + 8, ..., w + 56
#pragma unroll
    for (int kk = 0; kk < kDecodeSub / 8; ++kk) {
      const int key = warp + 8 * kk;
      float dot = 0.f;
      if (ok && key < nvalid) {
        if constexpr (kPerLane == 8) {
          const uint4 raw = *reinterpret_cast<const uint4*>(kst + key * (D * 2) + lane * 16);
          const float2 a = unpack2<BF16>(raw.x), b = unpack2<BF16>(raw.y);
          const float2 c = unpack2<BF16>(raw.z), e = unpack2<BF16>(raw.w);
          dot = qv[0] * a.x + qv[1] * a.y + qv[2] * b.x + qv[3] * b.y + qv[4] * c.x +
                qv[5] * c.y + qv[6] * e.x + qv[7] * e.y;
        } else if constexpr (kPerLane == 4) {
          const uint2 raw = *reinterpret_cast<const uint2*>(kst + key * (D * 2) + lane * 8);
          const float2 a = unpack2<BF16>(raw.x), b = unpack2<BF16>(raw.y);
          dot = qv[0] * a.x + qv[1] * a.y + qv[2] * b.x + qv[3] * b.y;
        } else {
          const float2 a =
              unpack2<BF16>(*reinterpret_cast<const uint32_t*>(kst + key * (D * 2) + lane * 4));
          dot = qv[0] * a.x + qv[1] * a.y;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      if (lane == 0) sc[key] = (key < nvalid) ? dot * p.scale_log2 : -INFINITY;
    }
    __syncthreads();
    // ---- running max, weights and sum (warp 0)
    if (warp == 0) {
      const float s0 = sc[lane], s1 = sc[lane + 32];
      float mb = fmaxf(s0, s1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
      const float m_new = fmaxf(m_run, mb);  // finite: a sub-block has >= 1 valid key
      const float alpha = ex2(m_run - m_new);
      const float p0 = ex2(s0 - m_new), p1 = ex2(s1 - m_new);
      pw[lane] = p0;
      pw[lane + 32] = p1;
      float ps = p0 + p1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l_run = l_run * alpha + ps;
      m_run = m_new;
      if (lane == 0) stat[0] = alpha;
    }
    __syncthreads();
    // ---- O~ = alpha O~ + sum_j p_j v_j over this thread's keys and column pair
    {
      const float alpha = stat[0];
      acc.x *= alpha;
      acc.y *= alpha;
      const int j0 = kg * kKeysPerGroup;
      const int j1 = min(j0 + kKeysPerGroup, nvalid);
      if (ok) {
        for (int j = j0; j < j1; ++j) {
          const float2 vv =
              unpack2<BF16>(*reinterpret_cast<const uint32_t*>(vst + j * (D * 2) + cp * 4));
          const float pj = pw[j];
          acc.x = fmaf(pj, vv.x, acc.x);
          acc.y = fmaf(pj, vv.y, acc.y);
        }
      }
    }
    __syncthreads();  // stage s, scores and weights are free again
    if (threadIdx.x == 0 && ok && i + NS < nsub) issue(i + NS);
  }

  // ---- join the key groups and write the split's record
  float* rec = p.partials + ((size_t)bh * p.splits + split) * C::kRecord;
  red[kg * D + 2 * cp] = acc.x;
  red[kg * D + 2 * cp + 1] = acc.y;
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += kDecodeThreads) {
    float u = 0.f;
#pragma unroll
    for (int g = 0; g < C::kGroups; ++g) u += red[g * D + c];
    rec[c] = (nsub > 0) ? u : 0.f;
  }
  if (threadIdx.x == 0) {
    rec[D] = (nsub > 0) ? m_run * kLn2 : -INFINITY;  // natural-log units
    rec[D + 1] = (nsub > 0) ? l_run : 0.f;
  }
  if (*abort_flag && threadIdx.x == 0) {
    // Copies this CTA started must land before its shared memory is released.
    for (int i = max(0, issued - NS); i < issued; ++i)
      mbar_wait(&full[i % NS], (i / NS) & 1, kDrainLimit, nullptr, kWaitDecDrain);
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_decode_merge_kernel(const float* partials,
                                                                 void* o, float* lse, int BH,
                                                                 int splits) {
  constexpr int kRecord = D + 4;
  constexpr int kCols = D / 32;  // columns per lane
  const int bh = blockIdx.x * 8 + warp_id();
  const int lane = lane_id();
  if (bh >= BH) return;
  const float* base = partials + (size_t)bh * splits * kRecord;
  float m = -INFINITY;
  for (int s = lane; s < splits; s += 32) m = fmaxf(m, base[(size_t)s * kRecord + D]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float l = 0.f;
  float u[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) u[c] = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float* rec = base + (size_t)s * kRecord;
    const float ms = rec[D];
    if (ms == -INFINITY) continue;  // empty split: the neutral state
    const float w = ex2((ms - m) * kLog2e);  // e^(m_s - m)
    l = fmaf(w, rec[D + 1], l);
    if constexpr (kCols == 8) {
      const float4 x = *reinterpret_cast<const float4*>(rec + lane * 8);
      const float4 y = *reinterpret_cast<const float4*>(rec + lane * 8 + 4);
      u[0] = fmaf(w, x.x, u[0]);
      u[1] = fmaf(w, x.y, u[1]);
      u[2] = fmaf(w, x.z, u[2]);
      u[3] = fmaf(w, x.w, u[3]);
      u[4] = fmaf(w, y.x, u[4]);
      u[5] = fmaf(w, y.y, u[5]);
      u[6] = fmaf(w, y.z, u[6]);
      u[7] = fmaf(w, y.w, u[7]);
    } else if constexpr (kCols == 4) {
      const float4 x = *reinterpret_cast<const float4*>(rec + lane * 4);
      u[0] = fmaf(w, x.x, u[0]);
      u[1] = fmaf(w, x.y, u[1]);
      u[2] = fmaf(w, x.z, u[2]);
      u[3] = fmaf(w, x.w, u[3]);
    } else {
      const float2 x = *reinterpret_cast<const float2*>(rec + lane * 2);
      u[0] = fmaf(w, x.x, u[0]);
      u[1] = fmaf(w, x.y, u[1]);
    }
  }
  const float inv = 1.f / l;
  uint8_t* orow = reinterpret_cast<uint8_t*>(o) + (size_t)bh * (D * 2);
  if constexpr (kCols == 8) {
    *reinterpret_cast<uint4*>(orow + lane * 16) =
        make_uint4(pack2<BF16>(u[0] * inv, u[1] * inv), pack2<BF16>(u[2] * inv, u[3] * inv),
                   pack2<BF16>(u[4] * inv, u[5] * inv), pack2<BF16>(u[6] * inv, u[7] * inv));
  } else if constexpr (kCols == 4) {
    *reinterpret_cast<uint2*>(orow + lane * 8) =
        make_uint2(pack2<BF16>(u[0] * inv, u[1] * inv), pack2<BF16>(u[2] * inv, u[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(orow + lane * 4) = pack2<BF16>(u[0] * inv, u[1] * inv);
  }
  if (lane == 0) lse[bh] = m + logf(l);
}

}  // namespace attn
