// fwd.cuh - attention forward on sm_103a: O = softmax(scale Q K^T [causal]) V and the
// per-row logsumexp L, with the online-softmax recurrence.
//
// Method ("Triton 05: Flash Attention", sections Online Softmax and 코드 라인별 설명
// (Forward); "FlashAttention·FA4·FP4", section 온라인 softmax가 블록 사이의 값을 어떻게
// 이어 주나): for each block of keys, S = scale Q K_j^T, m' = max(m, rowmax S),
// l' = exp(m - m') l + rowsum exp(S - m'), O' = exp(m - m') O + exp(S - m') V_j; after
// the last block O / l once, and L = m + ln l. The scores never leave the chip.
//
// GB300 design (the pages' kernels were written for A100 / Ada / B200: prior art):
//  * One CTA = one (b, h) slice x one 128-row query tile. Q_i is copied once from global
//    memory into tensor memory, so S = Q_i K_j^T is a TS product (A from tensor memory,
//    K_j from shared memory). On this part an MMA with both operands in shared memory
//    and N = 128 runs at about half the tensor rate (the tensor core's shared-memory
//    reads limit it); the TS form runs at the full rate.
//  * S is double buffered in tensor memory: the tensor core computes S_{j+1} (and P_j V_j)
//    while the softmax warps work on block j, in place of the two-tile ping-pong
//    described for Blackwell on "FlashAttention·FA4·FP4", section HBM을 아낀 뒤에는
//    무엇이 기다리는가. Tensor memory: S0, S1 (128 columns each), O (d), Q (d / 2).
//  * Warp roles: warps 0-7 softmax (warp w: rows 32 (w % 4) .. + 31 of the tile, score
//    columns 64 (w / 4) .. + 63 of each block), warp 8 TMA producer of the K ring, warp
//    10 of the V ring, warp 9 MMA issuer (one thread) and TMEM owner. The two warps that
//    share rows agree on the running max through shared memory and a two-arrival mbarrier
//    each block.
//  * Each K or V tile is one TMA copy (a 4-D view of the rows, see tma_load_tile), and K
//    and V have a producer thread each: what limits how fast one SM takes in tiles is the
//    round trip of the producer thread (wait for a free stage, issue), not the copy
//    engine, so fewer and larger copies from two threads keep the tensor core fed.
//  * P is written back over its own half of S as 16-bit pairs (columns [0, 32) and
//    [64, 96)) and fed to the P V product straight from tensor memory.
//  * exp is exp2 with scale*log2(e) folded into one FFMA per score ("Triton 05",
//    section 2. exp -> exp2 트릭); L is exported in the natural log.
//  * P is rounded to the input type for P V (the Triton code's p.to(v.dtype)). O is
//    divided by the sum of those same rounded values, so numerator and denominator use
//    one set of weights (the mismatch that "FlashAttention·FA4·FP4", FP4 section, warns
//    about); L uses the unrounded sum.
//  * The O rescale is conditional: the running max used for exp2 is only moved when
//    the row max grows by more than 8 (a factor 256), otherwise the stale max is kept
//    for both the numerator and l, which leaves O = acc / l exact ("FlashAttention·
//    FA4·FP4", section HBM을 아낀 뒤에는 무엇이 기다리는가, the rescale skip).
//  * Causal: key blocks after a tile's diagonal block are skipped; only the diagonal
//    block (and a ragged last block) is masked. The CTAs of one head are adjacent in
//    launch order (K/V of the head stay in L2) and run longest-first.
#pragma once

#include "common.cuh"

namespace attn {

struct FwdParams {
  const void* q;
  void* o;
  float* lse;
  int N;
  int nkb;          // number of 128-key blocks
  int nqt;          // number of 128-row query tiles
  int causal;
  float scale_log2; // scale * log2(e)
  unsigned long long wait_limit;
};

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / kBoxCols;            // 64-column boxes per row
  static constexpr int kTileBytes = kChunks * kBoxBytes;  // one 128 x D tile
  static constexpr int kStages = (D == 128) ? 3 : 4;      // depth of the K and V rings
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  // Exchange area: running-max halves [2 slots][2 halves][128 rows], then l and the
  // rounded sum [2][2 halves][128 rows] for the epilogue.
  static constexpr int kOffX = kOffV + kStages * kTileBytes;
  static constexpr int kXFloats = 2 * 2 * 128 + 2 * 2 * 128;
  static constexpr int kOffBar = kOffX + kXFloats * 4;
  // barriers: q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2],
  // o_done, o_last, pair[4], drain
  static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 2 + 4 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  // All 512 tensor-memory columns per CTA: one CTA per SM, which the shared memory
  // footprint (> 114 KiB for both head dims) already guarantees.
  static_assert(kSmemBytes > 114 * 1024, "two CTAs could share an SM");
  static constexpr int kThreads = 352;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColQ = 256 + D;
  static_assert(kColQ + D / 2 <= kTmemCols, "tensor memory overflow");
};

// Copies this thread's half row of Q (D / 2 16-bit values, D bytes) into tensor memory
// as 16-bit pairs; a null source (a row past the end) writes zeros.
template <int D>
__device__ __forceinline__ void copy_half_row_to_tmem(const uint8_t* src, uint32_t t_col) {
  constexpr int kWords = D / 4;  // 32-bit words in D bytes
  uint32_t r[kWords];
#pragma unroll
  for (int k = 0; k < kWords / 4; ++k) {
    const uint4 v = src ? *reinterpret_cast<const uint4*>(src + k * 16) : make_uint4(0, 0, 0, 0);
    r[4 * k] = v.x;
    r[4 * k + 1] = v.y;
    r[4 * k + 2] = v.z;
    r[4 * k + 3] = v.w;
  }
  if constexpr (kWords == 32) {
    tmem_st32(t_col, r);
  } else {
    tmem_st16(t_col, r);
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(352, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NS;
  uint64_t* v_full = k_empty + NS;
  uint64_t* v_empty = v_full + NS;
  uint64_t* s_full = v_empty + NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;  // each P_j V_j done (phase j)
  uint64_t* o_last = o_done + 1;  // all of them done (one phase)
  uint64_t* pair = o_last + 1;
  uint64_t* drain = pair + 4;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int bh = blockIdx.y;
  const int qt = p.nqt - 1 - blockIdx.x;  // within a head, longest (most key blocks) first
  const int q0 = qt * kTileM;
  const int N = p.N;
  const int n = p.causal ? min(p.nkb, qt + 1) : p.nkb;  // key blocks this tile needs

  if (threadIdx.x == 0) {
    mbar_init(q_full, 8);  // one arrival per softmax warp (its half rows of Q stored)
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 8);
    }
    mbar_init(o_done, 1);
    mbar_init(o_last, 1);
    for (int g = 0; g < 4; ++g) mbar_init(&pair[g], 2);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint64_t limit = p.wait_limit;

  if (warp == 8 || warp == 10) {
    // ------------------------------ TMA producers -----------------------------
    // Warp 8 fills the K ring, warp 10 the V ring, one whole-tile copy per block. The
    // warp runs converged (waits in every lane); the elected lane issues the copies.
    const bool is_k = warp == 8;
    const CUtensorMap* map = is_k ? &map_k : &map_v;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    uint8_t* ring = smem + (is_k ? C::kOffK : C::kOffV);
    if (elect_one()) tma_prefetch_map(map);
    int issued = 0;
    for (int i = 0; i < n; ++i) {
      const int s = i % NS;
      if (i >= NS &&
          !warp_wait(&empty[s], ((i / NS) - 1) & 1, limit, abort_flag, kWaitFwdEmpty))
        break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&full[s], C::kTileBytes);
        tma_load_tile(ring + s * C::kTileBytes, map, &full[s], i * kTileN, bh);
      }
      __syncwarp();
      issued = i + 1;
    }
    if (*abort_flag) {
      // Let every copy this warp started land before its shared memory is released.
      for (int g = max(0, issued - NS); g < issued; ++g)
        mbar_wait(&full[g % NS], (g / NS) & 1, limit, nullptr, kWaitFwdDrain);
    }
  } else if (warp == 9) {
    // ------------------------------ MMA issuer --------------------------------
    // The whole warp runs the loop and waits; one elected lane issues the MMAs and the
    // commits. Per block j: P_j V_j into O, then S_{j+2} into the buffer P_j came from (the
    // tensor core runs one thread's MMAs in issue order, so P_j is read first).
    const uint32_t idesc_s = make_idesc(BF16, 128, kTileN, false, false);
    const uint32_t idesc_o = make_idesc(BF16, 128, D, false, true);
    // Descriptors of stage 0 of each ring; stage s adds s * kTileBytes / 16.
    const uint64_t dk = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dv = make_sdesc_sw128(smem_u32(smem + C::kOffV), kBoxBytes, 1024);
    constexpr uint32_t kStageStep = C::kTileBytes >> 4;
    const uint32_t tq = tmem + C::kColQ;
    const uint32_t col_s[2] = {C::kColS0, C::kColS1};
    bool ok = warp_poll(q_full, 0, limit, abort_flag, kWaitFwdQ);
    for (int j = 0; ok && j < min(2, n); ++j) {
      const int s = j % NS;
      if (!(ok = warp_poll(&k_full[s], (j / NS) & 1, limit, abort_flag, kWaitFwdK))) break;
      tc_fence_after();
      if (elect_one()) {
        issue_rowdot_ts_d<D>(tmem + col_s[j], tq, dk + s * kStageStep, idesc_s);
        mma_commit(&s_full[j]);
        mma_commit(&k_empty[s]);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n; ++j) {
      const int b = j & 1;
      const int s = j % NS;
      if (!(ok = warp_poll(&v_full[s], (j / NS) & 1, limit, abort_flag, kWaitFwdV))) break;
      if (!(ok = warp_poll(&p_full[b], (j >> 1) & 1, limit, abort_flag, kWaitFwdP))) break;
      tc_fence_after();
      if (elect_one()) {
        issue_tmem_a_split_d(tmem + C::kColO, tmem + col_s[b], dv + s * kStageStep, idesc_o,
                             j > 0);
        mma_commit(o_done);
        mma_commit(&v_empty[s]);
      }
      __syncwarp();
      const int jn = j + 2;
      if (jn < n) {
        const int sn = jn % NS;
        if (!(ok = warp_poll(&k_full[sn], (jn / NS) & 1, limit, abort_flag, kWaitFwdK))) break;
        tc_fence_after();
        if (elect_one()) {
          issue_rowdot_ts_d<D>(tmem + col_s[b], tq, dk + sn * kStageStep, idesc_s);
          mma_commit(&s_full[b]);
          mma_commit(&k_empty[sn]);
        }
        __syncwarp();
      }
    }
    // The epilogue waits on its own barrier: when the softmax leaves its last block two
    // P V products can still be in flight, and a parity wait on o_done would then see the
    // phase before them as the one it waits for. Every MMA issued must finish before tensor
    // memory is released (drain).
    if (elect_one()) {
      if (ok) mma_commit(o_last);
      mma_commit(drain);
    }
    __syncwarp();
    mbar_wait(drain, 0, limit, nullptr, kWaitFwdDrain);
  } else {
    // ------------------------------ softmax -----------------------------------
    const int g = warp & 3;   // row group: tile rows [32 g, 32 g + 32)
    const int h = warp >> 2;  // column half: score columns [64 h, 64 h + 64)
    const uint32_t lane_base = (uint32_t)(g * 32) << 16;
    const int r = g * 32 + lane;  // row within the tile
    const int row = q0 + r;       // query index of this thread
    float* xm = reinterpret_cast<float*>(smem + C::kOffX);  // [2 slots][2 halves][128]
    float* xl = xm + 2 * 2 * 128;                            // [l, lr][2 halves][128]
    const float sl2 = p.scale_log2;

    // Q half row -> tensor memory (A operand of S = Q K^T).
    {
      const uint8_t* src =
          row < N ? reinterpret_cast<const uint8_t*>(p.q) +
                        ((size_t)bh * N + (size_t)row) * (size_t)(D * 2) + h * D
                  : nullptr;
      copy_half_row_to_tmem<D>(src, tmem + lane_base + C::kColQ + h * (D / 4));
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(q_full);
    }

    float m = -INFINITY;  // running max of scale*log2(e)*S (possibly stale by <= 8)
    float l = 0.f;        // sum of exp2 values over this warp's columns (fp32)
    float lr = 0.f;       // sum of the same values after rounding to 16 bits
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      const uint32_t t_s = tmem + lane_base + (b == 0 ? C::kColS0 : C::kColS1) + 64 * h;
      if (!(ok = warp_wait(&s_full[b], (j >> 1) & 1, limit, abort_flag, kWaitFwdS))) break;
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld64(t_s, sr);
      float* s = reinterpret_cast<float*>(sr);
      const int kbase = j * kTileN + 64 * h;  // key index of this warp's column 0
      if ((p.causal && kbase + 63 > q0) || kbase + 64 > N) {
        int lim = N - 1 - kbase;                    // last key in range
        if (p.causal) lim = min(lim, row - kbase);  // last key visible to this row
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      // Max over this warp's 64 columns in four independent chains of 3-input max.
      float mx[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) mx[u] = fmaxf(s[2 * u], s[2 * u + 1]);
#pragma unroll
      for (int c = 8; c < 64; c += 8) {
#pragma unroll
        for (int u = 0; u < 4; ++u) mx[u] = fmax3(mx[u], s[c + 2 * u], s[c + 2 * u + 1]);
      }
      const float m_half = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      // The row max over both halves: both warps compute the same value bit for bit.
      xm[(b * 2 + h) * 128 + r] = m_half;
      warp_arrive(&pair[g]);
      if (!(ok = warp_wait(&pair[g], j & 1, limit, abort_flag, kWaitFwdX))) break;
      const float m_cand = fmaxf(m_half, xm[(b * 2 + (h ^ 1)) * 128 + r]) * sl2;
      const bool need = m_cand > m + 8.0f;
      float alpha = 1.f;
      if (need) {
        alpha = ex2(m - m_cand);  // 0 on the first block (m = -inf)
        m = m_cand;
      }
      const float2 sl2x2 = make_float2(sl2, sl2);
      const float2 neg_m2 = make_float2(-m, -m);
      // l sums the fp32 values (it defines L); lr sums the 16-bit values that enter
      // P V, so that O = acc / lr divides by exactly the weights it accumulated.
      float2 sum[4];
      float rsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int u = 0; u < 4; ++u) sum[u] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c4 = 0; c4 < 2; ++c4) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x =
              fma2(make_float2(s[c4 * 32 + 2 * i], s[c4 * 32 + 2 * i + 1]), sl2x2, neg_m2);
          const float2 pp = make_float2(ex2(x.x), ex2(x.y));
          sum[i & 3] = add2(sum[i & 3], pp);
          pk[i] = pack2<BF16>(pp.x, pp.y);
          add_pair16<BF16>(rsum[(i & 1) * 2], rsum[(i & 1) * 2 + 1], pk[i]);
        }
        tmem_st16(t_s + c4 * 16, pk);
      }
      const float2 sa = add2(add2(sum[0], sum[1]), add2(sum[2], sum[3]));
      l = l * alpha + (sa.x + sa.y);
      lr = lr * alpha + ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3]));
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // Bring this warp's half of O to the new max once P_{j-1} V_{j-1} has landed
        // (P_{j-2} V_{j-2} has: S_j, already waited for, was issued after it).
        if (!(ok = warp_wait(o_done, (j - 1) & 1, limit, abort_flag, kWaitFwdO))) break;
        tc_fence_after();
        const uint32_t t_o = tmem + lane_base + C::kColO + h * (D / 2);
        if constexpr (D == 128) {
          uint32_t o[64];
          tmem_ld64(t_o, o);
#pragma unroll
          for (int i = 0; i < 64; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&o[0]);
          uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&o[32]);
          tmem_st32(t_o, lo);
          tmem_st32(t_o + 32, hi);
        } else {
          uint32_t o[32];
          tmem_ld32(t_o, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(t_o, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&p_full[b]);
    }
    if (ok) {
      // Both halves' sums, then this warp's half of the O row.
      xl[h * 128 + r] = l;
      xl[(2 + h) * 128 + r] = lr;
      warp_arrive(&pair[g]);
      ok = warp_wait(&pair[g], n & 1, limit, abort_flag, kWaitFwdX);
    }
    if (ok) {
      const float l_row = l + xl[(h ^ 1) * 128 + r];
      const float lr_row = lr + xl[(2 + (h ^ 1)) * 128 + r];
      ok = warp_wait(o_last, 0, limit, abort_flag, kWaitFwdO);
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.f / lr_row;
        const uint32_t t_o = tmem + lane_base + C::kColO + h * (D / 2);
        uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                        ((size_t)bh * N + (size_t)row) * (size_t)(D * 2) + h * D;
        constexpr int kCols = D / 2;  // fp32 columns of this half
        uint32_t o[kCols];
        if constexpr (kCols == 64) {
          tmem_ld64(t_o, o);
        } else {
          tmem_ld32(t_o, o);
        }
        uint32_t pk[kCols / 2];
#pragma unroll
        for (int i = 0; i < kCols / 2; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l,
                              __uint_as_float(o[2 * i + 1]) * inv_l);
        if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int v = 0; v < kCols / 8; ++v)
            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          if (h == 0) p.lse[(size_t)bh * N + row] = (m + log2f(l_row)) * kLn2;
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace attn
