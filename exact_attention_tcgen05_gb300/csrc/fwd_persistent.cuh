// fwd_persistent.cuh - the attention forward of fwd.cuh as a persistent kernel: one CTA per
// SM walks a list of work items (256 query rows of one (b, h) slice each) instead of one
// CTA per item.
//
// Why: a CTA of the one-item kernel pays a fixed cost of about 6 us (launch, barrier and
// tensor-memory set-up, the first Q/K/V copies from memory, the pipeline's first block, the
// epilogue) - measured on GB300 by timing whole waves of CTAs with 1 to 32 key blocks
// each, as much as three key blocks of work. Here the pipeline keeps running across
// items: the K/V ring, the barrier phases and the tensor memory carry over, the next
// item's Q is fetched as soon as the current item's last S = Q K^T has been issued, and
// the epilogue of one item (O / l from tensor memory to HBM) overlaps the first products
// of the next.
//
// The arithmetic of every item is exactly that of fwd.cuh (same tiles, same order, same
// rounding): the outputs are bit-identical.
//
// Schedule: items are numbered head by head, longest (most key blocks) first within a
// head, so the CTAs working at one time share the K/V of a few heads in L2. By default CTA
// c takes items c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... (G CTAs): a serpentine over the
// list, which pairs a long causal item of one round with a short one of the next. With
// few rounds of unequal causal items that leaves the busiest CTA well above the mean, so
// for dense causal inputs the host computes a longest-first greedy assignment instead
// (kernels_fwd.cu) and passes it as a table in the kernel's parameters.
//
// Barrier phases: every barrier completes once per event of a running count kept alike by
// all roles (blocks per tile, items per tile, Q loads, ring fills), and a wait names the
// parity of that count. No barrier can run two phases ahead of its waiter: each
// completion needs a step the waiter takes after its previous wait (the argument is given
// at each barrier below).
#pragma once

#include "fwd.cuh"
#include "schedule.h"

namespace attn {

// One work item: which rows, which keys, how many key blocks per tile.
struct FwdItem {
  SliceRows sl;
  int N, Nk, off;
  int q0;       // first query row of the item within its slice
  int nkv[2];   // key blocks of tile 0 / tile 1 (0: the tile lies past the slice's end)
  int n_kv;     // max of the two
};

// The k-th item of CTA c among G (serpentine order); -1 past the end.
__device__ __forceinline__ int fwd_item_index(int k, int G, int c, int n_items) {
  const int i = k * G + ((k & 1) ? (G - 1 - c) : c);
  return i < n_items ? i : -1;
}

// The schedule types the persistent kernel takes (by value, as a kernel parameter): the
// serpentine above, or an ItemTable (schedule.h).
struct FwdSerpentine {};
__device__ __forceinline__ int fwd_sched_item(const FwdSerpentine&, int k, int G, int c,
                                              int n_items) {
  return fwd_item_index(k, G, c, n_items);
}
__device__ __forceinline__ int fwd_sched_item(const ItemTable& t, int k, int, int c, int) {
  return table_item(t, k, c);
}

// Geometry of item `item` (nqb_max query blocks per slice). False: nothing to do (a packed
// sequence shorter than this block, or a malformed sequence, reported by slice_rows).
template <int D, bool PACKED>
__device__ __forceinline__ bool fwd_item_geom(const FwdParams& p, int item, int nqb_max,
                                              FwdItem& it) {
  const int bh = item / nqb_max;
  const int x = item - bh * nqb_max;
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, it.sl)) return false;
  it.N = it.sl.nq;
  it.Nk = it.sl.nk;
  it.off = it.sl.off;
  const int nqb = (it.N + 2 * kTileM - 1) / (2 * kTileM);
  if (x >= nqb) return false;
  const int nkb = (it.Nk + kTileN - 1) / kTileN;
  it.q0 = (nqb - 1 - x) * 256;  // within a head, longest first
  const int ntiles = (it.q0 + kTileM < it.N) ? 2 : 1;
#pragma unroll
  for (int t = 0; t < 2; ++t)
    it.nkv[t] = (t < ntiles)
                    ? (p.causal ? min(nkb, (it.q0 + t * kTileM + kTileM - 1 + it.off) / kTileN + 1)
                                : nkb)
                    : 0;
  it.n_kv = max(it.nkv[0], it.nkv[1]);
  return true;
}

template <int D>
struct FwdPCfg : FwdCfg<D> {
  using B = FwdCfg<D>;
  // The barriers of the one-item kernel, then q_empty and o_free[2].
  static constexpr int kNumBars = B::kNumBars + 3;
  static constexpr int kOffMisc = B::kOffBar + kNumBars * 8;
  // d = 64: each softmax warp stages its 32 rows of normalised O in shared memory (4 KiB,
  // 128-byte swizzle) and writes them with one TMA store, so the epilogue's global writes
  // run asynchronously instead of as 16-byte stores row by row (dense tensors; packed
  // batches keep the row stores, since a tile may run past its sequence into the next one's
  // rows).
  static constexpr bool kStageO = (D == 64);
  static constexpr int kOffO = ((kOffMisc + 16 + 1023) / 1024) * 1024;
  static constexpr int kSmemBytes = (kStageO ? kOffO + 2 * B::kTileBytes : kOffMisc + 16) + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

template <int D, bool BF16, bool PACKED, class Sched>
__global__ void __launch_bounds__(320, 1)
    attn_fwd_persistent_kernel(const __grid_constant__ CUtensorMap map_q,
                               const __grid_constant__ CUtensorMap map_k,
                               const __grid_constant__ CUtensorMap map_v,
                               const __grid_constant__ CUtensorMap map_o, const FwdParams p,
                               int n_items, int nqb_max, const __grid_constant__ Sched sched) {
  using C = FwdPCfg<D>;
  constexpr bool kTmaO = C::kStageO && !PACKED;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NS;
  uint64_t* kv_empty = v_full + NS;
  uint64_t* s_full = kv_empty + NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 2;
  uint64_t* s_free = drain + 1;   // [2] own-P layout: the softmax warps have read S_t
  uint64_t* q_empty = s_free + 2;  // the item's S products have all been issued and done
  uint64_t* o_free = q_empty + 1;  // [2] the epilogue has read O_t into registers
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);  // one arrival per softmax warp
      mbar_init(&o_done[t], 1);
      mbar_init(&s_free[t], 4);
      mbar_init(&o_free[t], 4);
    }
    mbar_init(drain, 1);
    mbar_init(q_empty, 1);
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
    if (elect_one()) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
    }
    __syncwarp();
    int q_loads = 0, kv_loads = 0;  // copies issued so far (running counts)
    for (int k = 0;; ++k) {
      const int item = fwd_sched_item(sched, k, G, cta, n_items);
      if (item < 0) break;
      FwdItem it;
      if (!fwd_item_geom<D, PACKED>(p, item, nqb_max, it)) continue;
      // Q of the previous item must have been read by every S product that uses it.
      // q_empty completes once per item after the item's last S; its next completion
      // needs the Q loaded below, so it is never two phases ahead of this wait.
      if (q_loads > 0 &&
          !warp_wait(q_empty, (q_loads - 1) & 1, limit, abort_flag, kWaitFwdQEmpty))
        break;
      const int ntiles = it.nkv[1] > 0 ? 2 : 1;
      if (elect_one()) {
        mbar_arrive_expect_tx(q_full, ntiles * C::kTileBytes);
        for (int t = 0; t < ntiles; ++t)
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_rows<PACKED>(smem + C::kOffQ + t * C::kTileBytes + c * kBoxBytes, &map_q,
                                  q_full, c * kBoxCols, it.q0 + t * kTileM, it.sl, false);
      }
      __syncwarp();
      ++q_loads;
      bool ok = true;
      for (int j = 0; j < it.n_kv; ++j) {
        const int s = kv_loads % NS;
        if (kv_loads >= NS &&
            !(ok = warp_wait(&kv_empty[s], ((kv_loads / NS) - 1) & 1, limit, abort_flag,
                             kWaitFwdEmpty)))
          break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&k_full[s], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_rows<PACKED>(smem + C::kOffK + s * C::kTileBytes + c * kBoxBytes, &map_k,
                                  &k_full[s], c * kBoxCols, j * kTileN, it.sl, true);
          mbar_arrive_expect_tx(&v_full[s], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_rows<PACKED>(smem + C::kOffV + s * C::kTileBytes + c * kBoxBytes, &map_v,
                                  &v_full[s], c * kBoxCols, j * kTileN, it.sl, true);
        }
        __syncwarp();
        ++kv_loads;
      }
      if (!ok) break;
    }
    if (*abort_flag) {
      // Let every copy this CTA started land before its shared memory is released.
      if (q_loads > 0) mbar_wait(q_full, (q_loads - 1) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
      for (int b = max(0, kv_loads - NS); b < kv_loads; ++b) {
        mbar_wait(&k_full[b % NS], (b / NS) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
        mbar_wait(&v_full[b % NS], (b / NS) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
      }
    }
  }
  else if (warp == 9) {
    // ------------------------------ MMA issuer --------------------------------
    const uint32_t idesc_s = make_idesc(BF16, 128, kTileN, false, false);
    const uint32_t idesc_o = make_idesc(BF16, 128, D, false, true);
    const uint64_t dq0 = make_sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t dk0 = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dv0 = make_sdesc_sw128(smem_u32(smem + C::kOffV), kBoxBytes, 1024);
    constexpr uint32_t kStep = C::kTileBytes >> 4;
    const uint32_t col_s[2] = {C::kColS0, C::kColS1};
    const uint32_t col_o[2] = {C::kColO0, C::kColO1};
    const uint32_t col_p[2] = {C::kOwnP ? C::kColP0 : C::kColS0,
                               C::kOwnP ? C::kColP1 : C::kColS1};
    auto issue_s = [&](int t, int stage) {
      issue_rowdot_d<D>(tmem + col_s[t], dq0 + t * kStep, dk0 + stage * kStep, idesc_s);
    };
    auto issue_pv = [&](int t, int stage, bool acc) {
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        mma_ts(tmem + col_o[t], tmem + col_p[t] + kk * 8,
               dv0 + stage * kStep + ((kk * 2048) >> 4), idesc_o, (acc || kk > 0) ? 1u : 0u);
    };
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) mma_commit(bar);
      __syncwarp();
    };
    // Running counts: Q loads consumed, ring blocks consumed, blocks and items per tile.
    int q_used = 0, kv_base = 0;
    int tb[2] = {0, 0}, ti[2] = {0, 0};
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = fwd_sched_item(sched, k, G, cta, n_items);
      if (item < 0) break;
      FwdItem it;
      if (!fwd_item_geom<D, PACKED>(p, item, nqb_max, it)) continue;
      const int n_kv = it.n_kv;
      if (!(ok = warp_wait(q_full, q_used & 1, limit, abort_flag, kWaitFwdQ))) break;
      ++q_used;
      if (!(ok = warp_wait(&k_full[kv_base % NS], (kv_base / NS) & 1, limit, abort_flag,
                           kWaitFwdK)))
        break;
      // First S of each tile. It overwrites S_t: at d = 128 the previous P over S_t was read
      // by a P V issued earlier (the tensor core runs them in order); in the own-P layout
      // the softmax must have read the tile's last S (s_free).
      #pragma unroll
      for (int t = 0; t < 2 && ok; ++t) {
        if (it.nkv[t] == 0) continue;
        if (C::kOwnP && tb[t] > 0 &&
            !(ok = warp_wait(&s_free[t], (tb[t] - 1) & 1, limit, abort_flag, kWaitFwdX)))
          break;
        tc_fence_after();
        if (elect_one()) {
          issue_s(t, kv_base % NS);
          mma_commit(&s_full[t]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (n_kv == 1) commit(q_empty);  // every S of the item issued
      for (int j = 0; ok && j < n_kv; ++j) {
        const int b = kv_base + j, bn = b + 1;
        const int s = b % NS, sn = bn % NS;
        const int jn = j + 1;
        if constexpr (C::kOwnP) {
          // S(t, j+1) for both tiles as soon as each softmax has read S(t, j).
          bool next_k_ready = false;
          #pragma unroll
      for (int t = 0; t < 2 && ok; ++t) {
            if (jn >= it.nkv[t]) continue;
            if (!next_k_ready) {
              if (!(ok = warp_wait(&k_full[sn], (bn / NS) & 1, limit, abort_flag, kWaitFwdK)))
                break;
              next_k_ready = true;
            }
            if (!(ok = warp_wait(&s_free[t], (tb[t] + j) & 1, limit, abort_flag, kWaitFwdX)))
              break;
            tc_fence_after();
            if (elect_one()) {
              issue_s(t, sn);
              mma_commit(&s_full[t]);
            }
            __syncwarp();
          }
          if (!ok) break;
          if (jn == n_kv - 1) commit(q_empty);
          if (!(ok = warp_wait(&v_full[s], (b / NS) & 1, limit, abort_flag, kWaitFwdV))) break;
          #pragma unroll
      for (int t = 0; t < 2 && ok; ++t) {
            if (j >= it.nkv[t]) continue;
            // The first P V of an item overwrites O_t: the epilogue of the tile's previous
            // item must have read it (o_free: one completion per item of the tile, each
            // after a P V issued past this wait).
            if (j == 0 && ti[t] > 0 &&
                !(ok = warp_wait(&o_free[t], (ti[t] - 1) & 1, limit, abort_flag,
                                 kWaitFwdOFree)))
              break;
            if (!(ok = warp_wait(&p_full[t], (tb[t] + j) & 1, limit, abort_flag, kWaitFwdP)))
              break;
            tc_fence_after();
            if (elect_one()) {
              issue_pv(t, s, j > 0);
              mma_commit(&o_done[t]);
            }
            __syncwarp();
          }
        } else {
          if (!(ok = warp_wait(&v_full[s], (b / NS) & 1, limit, abort_flag, kWaitFwdV))) break;
          tc_fence_after();
          bool next_k_ready = false;
          #pragma unroll
      for (int t = 0; t < 2 && ok; ++t) {
            if (j >= it.nkv[t]) continue;
            if (j == 0 && ti[t] > 0 &&
                !(ok = warp_wait(&o_free[t], (ti[t] - 1) & 1, limit, abort_flag,
                                 kWaitFwdOFree)))
              break;
            if (!(ok = warp_wait(&p_full[t], (tb[t] + j) & 1, limit, abort_flag, kWaitFwdP)))
              break;
            tc_fence_after();
            if (elect_one()) {
              issue_pv(t, s, j > 0);
              mma_commit(&o_done[t]);
            }
            __syncwarp();
            if (jn < it.nkv[t]) {
              if (!next_k_ready) {
                if (!(ok = warp_wait(&k_full[sn], (bn / NS) & 1, limit, abort_flag,
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
          if (ok && jn == n_kv - 1) commit(q_empty);
        }
        if (ok) commit(&kv_empty[s]);
      }
      kv_base += n_kv;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        tb[t] += it.nkv[t];
        ti[t] += it.nkv[t] > 0 ? 1 : 0;
      }
    }
    // Every MMA issued must finish before tensor memory is released.
    commit(drain);
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitFwdDrain);
  }
  else {
    // ------------------------------ softmax (tile t) --------------------------
    const int t = warp >> 2;
    const int wq = warp & 3;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + (t == 0 ? C::kColS0 : C::kColS1);
    const uint32_t t_o = tmem + lane_base + (t == 0 ? C::kColO0 : C::kColO1);
    const uint32_t t_p = C::kOwnP ? tmem + lane_base + (t == 0 ? C::kColP0 : C::kColP1) : t_s;
    const float sl2 = p.scale_log2;
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
    int tb = 0;  // blocks of this tile so far (running count, as the MMA warp keeps it)
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = fwd_sched_item(sched, k, G, cta, n_items);
      if (item < 0) break;
      FwdItem it;
      if (!fwd_item_geom<D, PACKED>(p, item, nqb_max, it)) continue;
      // (a select, not it.nkv[t]: a runtime index would put the whole item in local memory)
      const int nkv = t == 0 ? it.nkv[0] : it.nkv[1];
      if (nkv == 0) continue;  // this tile lies past the slice's end
      const int row = it.q0 + t * kTileM + wq * 32 + lane;  // query index of this thread
      const int tile_row0 = it.q0 + t * kTileM;
      float m = -INFINITY;  // running max of scale*log2(e)*S (possibly stale by <= 8)
      float l = 0.f;        // sum of exp2 values (fp32)
      float lr = 0.f;       // sum of the same values after rounding to 16 bits
      for (int j = 0; j < nkv; ++j) {
        const int b = tb + j;
        if (!(ok = warp_wait(&s_full[t], b & 1, limit, abort_flag, kWaitFwdS))) break;
        tc_fence_after();
        uint32_t sr[kTileN];
        tmem_ld128(t_s, sr);
        if constexpr (C::kOwnP) {
          tc_fence_before();
          warp_arrive(&s_free[t]);  // S(t, j) is in registers: the next S may overwrite it
        }
        float* sv = reinterpret_cast<float*>(sr);
        const int kbase = j * kTileN;
        const bool diag = p.causal && (kbase + kTileN - 1 > tile_row0 + it.off);
        if (diag || kbase + kTileN > it.Nk) {
          int lim = it.Nk - 1 - kbase;                         // last key in range
          if (p.causal) lim = min(lim, row + it.off - kbase);  // last key this row sees
#pragma unroll
          for (int c = 0; c < kTileN; ++c)
            if (c > lim) sv[c] = -INFINITY;
        }
        float mx[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) mx[u] = fmaxf(sv[2 * u], sv[2 * u + 1]);
#pragma unroll
        for (int c = 8; c < kTileN; c += 8) {
#pragma unroll
          for (int u = 0; u < 4; ++u) mx[u] = fmax3(mx[u], sv[c + 2 * u], sv[c + 2 * u + 1]);
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
        float2 sum[4];
        float rsum[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pall[C::kOwnP ? kTileN / 2 : 1];
#pragma unroll
        for (int u = 0; u < 4; ++u) sum[u] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c4 = 0; c4 < kTileN / 32; ++c4) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = fma2(make_float2(sv[c4 * 32 + 2 * i], sv[c4 * 32 + 2 * i + 1]),
                                  sl2x2, neg_m2);
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
        l = l * alpha + (sa.x + sa.y);
        lr = lr * alpha + ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3]));
        if constexpr (C::kOwnP) {
          // The previous block's P V reads P_t and accumulates into O_t.
          if (j > 0) {
            if (!(ok = warp_wait(&o_done[t], (b - 1) & 1, limit, abort_flag, kWaitFwdO)))
              break;
            tc_fence_after();
            if (__any_sync(0xffffffffu, need)) rescale_o(alpha);
          }
#pragma unroll
          for (int c4 = 0; c4 < kTileN / 32; ++c4)
            tmem_st16(t_p + c4 * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pall[c4 * 16]));
        } else if (j > 0 && __any_sync(0xffffffffu, need)) {
          if (!(ok = warp_wait(&o_done[t], (b - 1) & 1, limit, abort_flag, kWaitFwdO))) break;
          tc_fence_after();
          rescale_o(alpha);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&p_full[t]);
      }
      if (!ok) break;
      // Epilogue: O_t of the last P V into registers, release O_t (o_free) so the next
      // item's first P V may overwrite it, then O / l and L to global memory.
      if (!(ok = warp_wait(&o_done[t], (tb + nkv - 1) & 1, limit, abort_flag, kWaitFwdO)))
        break;
      tc_fence_after();
      uint32_t r[D];
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc)
        tmem_ld64(t_o + cc * 64, *reinterpret_cast<uint32_t(*)[64]>(&r[cc * 64]));
      tc_fence_before();
      warp_arrive(&o_free[t]);
      tb += nkv;
      if constexpr (kTmaO) {
        // Each warp stages its 32 rows of O / l in a 4 KiB buffer of its own (128-byte
        // swizzle) and its lane 0 stores them with one TMA copy: no barrier beyond the warp.
        // The buffer's previous store must have read it first.
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        const float inv_l = 1.f / lr;
        uint8_t* buf = smem + C::kOffO + (t * 4 + wq) * 4096;
        const uint32_t rbase = smem_u32(buf) + lane * 128;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint32_t w4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            w4[i] = pack2<BF16>(__uint_as_float(r[8 * v + 2 * i]) * inv_l,
                                __uint_as_float(r[8 * v + 2 * i + 1]) * inv_l);
          st_shared_v4(rbase + ((v ^ (lane & 7)) << 4), w4[0], w4[1], w4[2], w4[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&map_o, buf, 0, tile_row0 + wq * 32, it.sl.tma_bh);
          bulk_commit_group();
        }
        if (row < it.N) p.lse[it.sl.stat0 + row] = (m + log2f(l)) * kLn2;
      } else if (row < it.N) {
        const float inv_l = 1.f / lr;
        uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                        (it.sl.q_elem0 + (size_t)row * it.sl.row_elems) * 2;
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            pk[i] = pack2<BF16>(__uint_as_float(r[cc * 64 + 2 * i]) * inv_l,
                                __uint_as_float(r[cc * 64 + 2 * i + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 128);
          const int n16 = valid16(p.dh, cc * 64, 8);  // columns past dh are not stored
#pragma unroll
          for (int v = 0; v < 8; ++v)
            if (v < n16)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
        p.lse[it.sl.stat0 + row] = (m + log2f(l)) * kLn2;
      }
    }
    // the warp's last store must have finished with its buffer before shared memory is
    // released
    if (kTmaO && lane == 0) bulk_wait_all();
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
