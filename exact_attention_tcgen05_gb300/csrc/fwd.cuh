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
//  * One CTA = one (b, h) slice x 256 query rows, split into two 128-row tiles that
//    ping-pong: while one tile's softmax runs on the CUDA cores, the tensor core works
//    on the other tile (the two-tile schedule described for Blackwell on
//    "FlashAttention·FA4·FP4", section HBM을 아낀 뒤에는 무엇이 기다리는가).
//  * Warp roles: warps 0-3 softmax of tile 0, warps 4-7 softmax of tile 1, warp 8 TMA
//    producer, warp 9 MMA issuer (one thread) and TMEM owner.
//  * Q tiles, and a ring of K/V blocks, are TMA-copied into 128B-swizzled shared
//    memory; S = Q K^T and O += P V run on tcgen05 with fp32 accumulators in tensor
//    memory (S_t: 128 columns, O_t: d columns per tile). P is written back over S_t as
//    16-bit pairs and fed to the P V product straight from tensor memory.
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
  const void* q;    // Q, for kernels that read its rows directly (the one-tile 256-column one)
  void* o;
  float* lse;
  int dh;           // head dimension of the tensors (<= D; columns past it read as zero)
  int N;            // query rows per slice (N_q; packed batches: per sequence, from vl)
  int Nk;           // key rows per slice (N_k)
  int causal;
  float scale_log2; // scale * log2(e)
  unsigned long long wait_limit;
  int stall;        // failure tests: the TMA producer withholds every copy
  Varlen vl;        // packed variable-length batch (vl.cu_q == nullptr: dense)
};

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / kBoxCols;            // 64-column boxes per row
  static constexpr int kTileBytes = kChunks * kBoxBytes;  // one 128 x D tile
  static constexpr int kStages = (D == 128) ? 2 : 4;      // K/V ring depth
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // barriers: q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], p_full[2],
  // o_done[2], drain, s_free[2]
  static constexpr int kNumBars = 1 + 3 * kStages + 6 + 1 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  // All 512 tensor-memory columns per CTA: one CTA per SM, which the shared memory
  // footprint (> 114 KiB for both head dims) already guarantees.
  static_assert(kSmemBytes > 114 * 1024, "two CTAs could share an SM");
  static constexpr int kThreads = 320;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  // d = 64: P gets tensor-memory columns of its own (S0 S1 O0 O1 P0 P1 fill the 512), so
  // S of the next key block is computed while the softmax still works on this one: it
  // waits only until the softmax warps have read S into registers (s_free), not for P V.
  // At d = 128 S and O fill all 512 columns and P is written over S.
  static constexpr bool kOwnP = (D == 64);
  static constexpr uint32_t kColP0 = 256 + 2 * D, kColP1 = 256 + 2 * D + 64;
};

template <int D, bool BF16, bool PACKED>
__global__ void __launch_bounds__(320, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + C::kStages;
  uint64_t* kv_empty = v_full + C::kStages;
  uint64_t* s_full = kv_empty + C::kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 2;
  uint64_t* s_free = drain + 1;  // [2]: the softmax warps have read S_t (own-P layout)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int bh = blockIdx.y;
  SliceRows sl;
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, sl)) return;
  const int N = sl.nq, Nk = sl.nk, off = sl.off;
  const int nqb = (N + 2 * kTileM - 1) / (2 * kTileM);
  const int nkb = (Nk + kTileN - 1) / kTileN;
  if (PACKED && (int)blockIdx.x >= nqb) return;  // past this sequence's query blocks
  const int qb = nqb - 1 - blockIdx.x;  // within a head, longest (most key blocks) first
  const int q0 = qb * 256;
  const int ntiles = (q0 + kTileM < N) ? 2 : 1;
  int nkv[2];
  for (int t = 0; t < 2; ++t) {
    // causal: up to the block of the last key the tile's last row sees
    nkv[t] = (t < ntiles) ? (p.causal ? min(nkb, (q0 + t * kTileM + kTileM - 1 + off) / kTileN + 1)
                                      : nkb)
                          : 0;
  }
  const int n_kv = max(nkv[0], nkv[1]);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);  // one arrival per softmax warp
      mbar_init(&o_done[t], 1);
      mbar_init(&s_free[t], 4);  // one arrival per softmax warp
    }
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

  if (warp == 8 && p.stall) {
    // Failure tests: the producer withholds every copy; the consumers' waits run out.
  } else if (warp == 8) {
    // ------------------------------ TMA producer ------------------------------
    // Converged warp (waits in every lane); the elected lane issues the copies.
    if (elect_one()) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      mbar_arrive_expect_tx(q_full, ntiles * C::kTileBytes);
      for (int t = 0; t < ntiles; ++t)
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffQ + t * C::kTileBytes + c * kBoxBytes, &map_q,
                                q_full, c * kBoxCols, q0 + t * kTileM, sl, false);
    }
    __syncwarp();
    int issued = 0;
    for (int j = 0; j < n_kv; ++j) {
      const int s = j % C::kStages;
      if (j >= C::kStages &&
          !warp_wait(&kv_empty[s], ((j / C::kStages) - 1) & 1, limit, abort_flag,
                     kWaitFwdEmpty))
        break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&k_full[s], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffK + s * C::kTileBytes + c * kBoxBytes, &map_k,
                                &k_full[s], c * kBoxCols, j * kTileN, sl, true);
        mbar_arrive_expect_tx(&v_full[s], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffV + s * C::kTileBytes + c * kBoxBytes, &map_v,
                                &v_full[s], c * kBoxCols, j * kTileN, sl, true);
      }
      __syncwarp();
      issued = j + 1;
    }
    if (*abort_flag) {
      // Let every copy this CTA started land before its shared memory is released.
      mbar_wait(q_full, 0, kDrainLimit, nullptr, kWaitFwdDrain);
      for (int j = max(0, issued - C::kStages); j < issued; ++j) {
        const int s = j % C::kStages;
        mbar_wait(&k_full[s], (j / C::kStages) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
        mbar_wait(&v_full[s], (j / C::kStages) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
      }
    }
  } else if (warp == 9) {
    // ------------------------------ MMA issuer --------------------------------
    // Converged warp; the elected lane issues the MMAs and commits.
    const uint32_t idesc_s = make_idesc(BF16, 128, kTileN, false, false);
    const uint32_t idesc_o = make_idesc(BF16, 128, D, false, true);
    const uint64_t dq0 = make_sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t dk0 = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dv0 = make_sdesc_sw128(smem_u32(smem + C::kOffV), kBoxBytes, 1024);
    constexpr uint32_t kStep = C::kTileBytes >> 4;
    const uint32_t col_s[2] = {C::kColS0, C::kColS1};
    const uint32_t col_o[2] = {C::kColO0, C::kColO1};
    const uint32_t col_p[2] = {C::kOwnP ? C::kColP0 : C::kColS0,
                               C::kOwnP ? C::kColP1 : C::kColS1};  // P: own columns or over S
    auto issue_s = [&](int t, int stage) {
      issue_rowdot_d<D>(tmem + col_s[t], dq0 + t * kStep, dk0 + stage * kStep, idesc_s);
    };
    auto issue_pv = [&](int t, int stage, bool acc) {
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        mma_ts(tmem + col_o[t], tmem + col_p[t] + kk * 8,
               dv0 + stage * kStep + ((kk * 2048) >> 4), idesc_o, (acc || kk > 0) ? 1u : 0u);
    };

    bool ok = warp_wait(q_full, 0, limit, abort_flag, kWaitFwdQ);
    if (ok) ok = warp_wait(&k_full[0], 0, limit, abort_flag, kWaitFwdK);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        for (int t = 0; t < 2; ++t)
          if (nkv[t] > 0) {
            issue_s(t, 0);
            mma_commit(&s_full[t]);
          }
      }
      __syncwarp();
    }
    if constexpr (C::kOwnP) {
      // Per key block j: S(t, j+1) for both tiles as soon as each softmax has read S(t, j),
      // then P(t, j) V_j as each P is ready.
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % C::kStages;
        const int jn = j + 1;
        const int sn = jn % C::kStages;
        bool next_k_ready = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if (jn >= nkv[t]) continue;
          if (!next_k_ready) {
            if (!(ok = warp_wait(&k_full[sn], (jn / C::kStages) & 1, limit, abort_flag,
                                 kWaitFwdK)))
              break;
            next_k_ready = true;
          }
          if (!(ok = warp_wait(&s_free[t], j & 1, limit, abort_flag, kWaitFwdX))) break;
          tc_fence_after();
          if (elect_one()) {
            issue_s(t, sn);
            mma_commit(&s_full[t]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (!(ok = warp_wait(&v_full[s], (j / C::kStages) & 1, limit, abort_flag, kWaitFwdV)))
          break;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= nkv[t]) continue;
          if (!(ok = warp_wait(&p_full[t], j & 1, limit, abort_flag, kWaitFwdP))) break;
          tc_fence_after();
          if (elect_one()) {
            issue_pv(t, s, j > 0);
            mma_commit(&o_done[t]);
          }
          __syncwarp();
        }
        if (ok) {
          if (elect_one()) mma_commit(&kv_empty[s]);
          __syncwarp();
        }
      }
    } else {
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % C::kStages;
        if (!(ok = warp_wait(&v_full[s], (j / C::kStages) & 1, limit, abort_flag, kWaitFwdV)))
          break;
        tc_fence_after();
        const int jn = j + 1;
        const int sn = jn % C::kStages;
        bool next_k_ready = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= nkv[t]) continue;
          if (!(ok = warp_wait(&p_full[t], j & 1, limit, abort_flag, kWaitFwdP))) break;
          tc_fence_after();
          if (elect_one()) {
            issue_pv(t, s, j > 0);
            mma_commit(&o_done[t]);
          }
          __syncwarp();
          if (jn < nkv[t]) {
            if (!next_k_ready) {
              if (!(ok = warp_wait(&k_full[sn], (jn / C::kStages) & 1, limit, abort_flag,
                                   kWaitFwdK)))
                break;
              tc_fence_after();
              next_k_ready = true;
            }
            if (elect_one()) {
              issue_s(t, sn);
              mma_commit(&s_full[t]);
            }
            __syncwarp();
          }
        }
        if (ok) {
          if (elect_one()) mma_commit(&kv_empty[s]);
          __syncwarp();
        }
      }
    }
    // Every MMA issued must finish before tensor memory is released.
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitFwdDrain);
  } else {
    // ------------------------------ softmax (tile t) --------------------------
    const int t = warp >> 2;
    const int wq = warp & 3;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + (t == 0 ? C::kColS0 : C::kColS1);
    const uint32_t t_o = tmem + lane_base + (t == 0 ? C::kColO0 : C::kColO1);
    const uint32_t t_p = C::kOwnP ? tmem + lane_base + (t == 0 ? C::kColP0 : C::kColP1) : t_s;
    const int row = q0 + t * kTileM + wq * 32 + lane;  // query index of this thread
    const int tile_row0 = q0 + t * kTileM;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running max of scale*log2(e)*S (possibly stale by <= 8)
    float l = 0.f;        // sum of exp2 values (fp32)
    float lr = 0.f;       // sum of the same values after rounding to 16 bits
    bool ok = true;
    // O *= alpha in tensor memory (the previous P V product must have landed).
    auto rescale_o = [&](float alpha) {
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t r[64];
        tmem_ld64(t_o + cc * 64, r);
#pragma unroll
        for (int i = 0; i < 64; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
        tmem_st32(t_o + cc * 64, lo);
        tmem_st32(t_o + cc * 64 + 32, hi);
      }
    };
    for (int j = 0; j < nkv[t]; ++j) {
      if (!(ok = warp_wait(&s_full[t], j & 1, limit, abort_flag, kWaitFwdS))) break;
      tc_fence_after();
      // One wide load of the whole score row, then a single wait.
      uint32_t sr[kTileN];
      tmem_ld128(t_s, sr);
      if constexpr (C::kOwnP) {
        tc_fence_before();
        warp_arrive(&s_free[t]);  // S(t, j) is in registers: S(t, j + 1) may overwrite it
      }
      float* s = reinterpret_cast<float*>(sr);
      const int kbase = j * kTileN;
      const bool diag = p.causal && (kbase + kTileN - 1 > tile_row0 + off);
      if (diag || kbase + kTileN > Nk) {
        int lim = Nk - 1 - kbase;                       // last key in range
        if (p.causal) lim = min(lim, row + off - kbase);  // last key visible to this row
#pragma unroll
        for (int c = 0; c < kTileN; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      // Row max in four independent chains of 3-input max (short dependency chains).
      float mx[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) mx[u] = fmaxf(s[2 * u], s[2 * u + 1]);  // columns 0..7
#pragma unroll
      for (int c = 8; c < kTileN; c += 8) {  // columns 8..127
#pragma unroll
        for (int u = 0; u < 4; ++u) mx[u] = fmax3(mx[u], s[c + 2 * u], s[c + 2 * u + 1]);
      }
      const float m_cand = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
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
      // Two sums, each in four independent packed accumulators.
      float2 sum[4];
      float rsum[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pall[C::kOwnP ? kTileN / 2 : 1];  // own-P layout: all of P before the store
#pragma unroll
      for (int u = 0; u < 4; ++u) sum[u] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c4 = 0; c4 < kTileN / 32; ++c4) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x = fma2(make_float2(s[c4 * 32 + 2 * i], s[c4 * 32 + 2 * i + 1]), sl2x2,
                                neg_m2);
          const float2 pp = make_float2(ex2(x.x), ex2(x.y));
          sum[i & 3] = add2(sum[i & 3], pp);
          pk[i] = pack2<BF16>(pp.x, pp.y);
          add_pair16<BF16>(rsum[(i & 1) * 2], rsum[(i & 1) * 2 + 1], pk[i]);
        }
        if constexpr (C::kOwnP) {
#pragma unroll
          for (int i = 0; i < 16; ++i) pall[c4 * 16 + i] = pk[i];
        } else {
          tmem_st16(t_s + c4 * 16, pk);
        }
      }
      const float2 sa = add2(add2(sum[0], sum[1]), add2(sum[2], sum[3]));
      const float sum0 = sa.x, sum1 = sa.y, rsum0 = rsum[0] + rsum[1], rsum1 = rsum[2] + rsum[3];
      l = l * alpha + (sum0 + sum1);
      lr = lr * alpha + (rsum0 + rsum1);
      if constexpr (C::kOwnP) {
        // P V of the previous block reads P_t and accumulates into O_t: it must have
        // finished before P_t is overwritten or O_t rescaled.
        if (j > 0) {
          if (!(ok = warp_wait(&o_done[t], (j - 1) & 1, limit, abort_flag, kWaitFwdO))) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, need)) rescale_o(alpha);
        }
#pragma unroll
        for (int c4 = 0; c4 < kTileN / 32; ++c4)
          tmem_st16(t_p + c4 * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pall[c4 * 16]));
      } else if (j > 0 && __any_sync(0xffffffffu, need)) {
        // Bring O to the new max: wait until the previous P V product has landed.
        if (!(ok = warp_wait(&o_done[t], (j - 1) & 1, limit, abort_flag, kWaitFwdO))) break;
        tc_fence_after();
        rescale_o(alpha);
      }
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&p_full[t]);
    }
    if (ok && nkv[t] > 0 &&
        warp_wait(&o_done[t], (nkv[t] - 1) & 1, limit, abort_flag, kWaitFwdO)) {
      tc_fence_after();
      const float inv_l = 1.f / lr;
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                      (sl.q_elem0 + (size_t)row * sl.row_elems) * 2;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t r[64];
        tmem_ld64(t_o + cc * 64, r);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * inv_l,
                              __uint_as_float(r[2 * i + 1]) * inv_l);
        if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 128);
          const int n16 = valid16(p.dh, cc * 64, 8);  // columns past dh are not stored
#pragma unroll
          for (int v = 0; v < 8; ++v)
            if (v < n16)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (row < N) p.lse[sl.stat0 + row] = (m + log2f(l)) * kLn2;
    }
    tc_fence_before();
  }

  tmem_st_wait();  // no tensor-memory store in flight when memory is released
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace attn
