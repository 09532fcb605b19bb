// fwd_pair.cuh - the persistent attention forward of fwd_persistent.cuh on CTA pairs: two
// CTAs on two SMs (a cluster of two) share every key block, and the pair's products are
// tcgen05 MMAs with .cta_group::2 (M = 256 query rows, 128 in each CTA).
//
// What the pairing changes: each CTA holds half of the B operand of each product - keys
// [64r, 64r + 64) of K_j for S, columns [64r, 64r + 64) of V_j for P V (r = the CTA's rank)
// - so a key block costs each SM 32 KiB of copies instead of 64, and each SM's tensor core
// reads half as much B from shared memory per product. The method is that of fwd.cuh;
// only the distribution of the work changes (the pages' Blackwell kernel,
// "FlashAttention·FA4·FP4", section HBM을 아낀 뒤에는 무엇이 기다리는가, pairs SMs this way
// for its backward). Measured on GB300 it is slower than the one-CTA forward (B4 H32 N4096
// causal: 0.574 against 0.420 ms): the forward is bound by each tile's chain S -> softmax
// -> P V, and the pair adds the wait for the other CTA's P to it. The launcher runs it only
// on request (ATTN_FWD_PAIR = 1).
//
// Work: an item is 512 query rows (four 128-row blocks) of one (b, h) slice. Tile t
// (t = 0, 1) of the pair is the 256 rows [q0 + 256t, q0 + 256t + 256); CTA r holds rows
// [q0 + 256t + 128r, +128) of it in shared memory (its Q_t) and gets their S_t and O_t in
// its tensor memory. Key block j: CTA r loads K_j rows [64r, 64r + 64) (all d columns) and
// V_j columns [64r, 64r + 64) (all 128 keys). Causal: a tile's key blocks are those its
// last row sees; the rows of rank 0 mask the extra diagonal block (at most one per tile).
//
// Roles (the same in both CTAs unless stated): warps 0-3 / 4-7 the softmax of tile 0 / 1
// for this CTA's 128 rows; warp 8 the TMA producer of this CTA's halves; warp 9: in rank 0
// the MMA issuer (one elected lane), in rank 1 a forwarder that tells rank 0 when rank 1's
// copies have landed.
//
// Pair protocol (every wait bounded, as in the one-CTA kernels):
//  * Set-up: thread 0 initialises the barriers; warp 9 of each CTA allocates all 512
//    tensor-memory columns with tcgen05.alloc.cta_group::2 (one warp in each CTA of the
//    pair); then all threads of both CTAs meet at barrier.cluster (no remote access happens
//    before it). Rank 0 addresses both CTAs' tensor memory with its own column address, so
//    each CTA checks that the peer's allocation starts at the same address and otherwise
//    records kErrPairTmem and does no work.
//  * Copies: each CTA's TMA copies complete on its OWN barriers (q_full, k_full[s],
//    v_full[s]), with its own expect_tx; rank 1's warp 9 waits for each of them in the
//    order they were issued and then arrives (release, cluster scope) on rank 0's q_pfull,
//    k_pfull[s], v_pfull[s]. Rank 0's MMA warp waits for both its own and the forwarded
//    barrier before a product reads the stage. A CTA therefore only ever waits for its own
//    copies when it drains.
//  * Products: rank 0 issues every MMA and every tcgen05.commit with .cta_group::2; the
//    commits multicast to both CTAs (mask 0b11): s_full[t], o_done[t] (the softmax warps of
//    both CTAs read their own S_t / O_t), kv_empty[s], q_empty (both producers refill their
//    own slots) and drain.
//  * Results back: each CTA's softmax warps write P_t into their own tensor memory and
//    arrive (release, cluster scope) on rank 0's p_full[t] (8 warps: 4 per CTA); the
//    epilogue warps arrive on rank 0's o_free[t] once O_t is in registers. Rank 0 waits for
//    these with cluster-scope acquire.
//  * Exit: every role of a CTA ends (rank 0's MMA warp after its drain commit has landed,
//    rank 1's warp 9 after the same multicast drain has reached it, the producers after
//    their own copies after an abort), then thread 0 of each CTA arrives on the peer's exit
//    barrier and waits (bounded) for the peer's arrival on its own, and only then is the
//    tensor memory freed (tcgen05.dealloc.cta_group::2 in both CTAs) and the CTA ends. No
//    CTA leaves while the other can still touch its shared or tensor memory.
//
// The arithmetic of every row is that of fwd.cuh: the same products (the pair computes
// each S and P V element from the same operands in the same order), the same softmax and
// rounding.
#pragma once

#include "fwd_persistent.cuh"
#include "pair.cuh"

namespace attn {

template <int D>
struct FwdPairCfg {
  static_assert(D == 128, "the pair forward is built for 128-column heads");
  static constexpr int kQTileBytes = 2 * kBoxBytes;     // 128 rows x 128 columns
  static constexpr int kKHalfBytes = 2 * kBoxBytes / 2;  // 64 rows x 128 columns
  static constexpr int kVHalfBytes = kBoxBytes;          // 128 rows x 64 columns
  static constexpr int kKChunkBytes = kBoxBytes / 2;     // 64 rows x 64 columns
  static constexpr int kStages = 4;                      // key blocks in flight
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTileBytes;
  static constexpr int kOffV = kOffK + kStages * kKHalfBytes;
  static constexpr int kOffBar = kOffV + kStages * kVHalfBytes;
  // q_full, q_pfull, k_full[S], v_full[S], k_pfull[S], v_pfull[S], kv_empty[S], q_empty,
  // s_full[2], p_full[2], o_done[2], o_free[2], drain, exit
  static constexpr int kNumBars = 2 + 5 * kStages + 1 + 8 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kSmemBytes > 114 * 1024, "two CTAs could share an SM");
  static constexpr int kThreads = 320;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
};

// One pair item (the same in both CTAs): rows [q0, q0 + 512) of one slice.
struct FwdPairItem {
  SliceRows sl;
  int N, Nk, off;
  int q0;
  int nkv[2];  // key blocks of tile 0 / 1 (0: the tile lies past the slice's end)
  int n_kv;
};

template <bool PACKED>
__device__ __forceinline__ bool fwd_pair_item_geom(const FwdParams& p, int item, int nsb_max,
                                                   FwdPairItem& it) {
  const int bh = item / nsb_max;
  const int x = item - bh * nsb_max;
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, it.sl)) return false;
  it.N = it.sl.nq;
  it.Nk = it.sl.nk;
  it.off = it.sl.off;
  const int nsb = (it.N + 4 * kTileM - 1) / (4 * kTileM);
  if (x >= nsb) return false;
  const int nkb = (it.Nk + kTileN - 1) / kTileN;
  it.q0 = (nsb - 1 - x) * 4 * kTileM;  // within a head, longest first
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = it.q0 + t * 2 * kTileM;
    const int last = min(r0 + 2 * kTileM, it.N) - 1;  // the tile's last row in the slice
    it.nkv[t] = r0 >= it.N ? 0 : (p.causal ? min(nkb, (last + it.off) / kTileN + 1) : nkb);
  }
  it.n_kv = max(it.nkv[0], it.nkv[1]);
  return true;
}

template <bool BF16, bool PACKED, class Sched>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k64,
                         const __grid_constant__ CUtensorMap map_v, const FwdParams p,
                         int n_items, int nsb_max, const __grid_constant__ Sched sched) {
  constexpr int D = 128;
  using C = FwdPairCfg<D>;
  constexpr int NS = C::kStages;
  constexpr uint16_t kBoth = 0x3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_pfull = q_full + 1;   // rank 0: rank 1's Q copies have landed
  uint64_t* k_full = q_pfull + 1;   // [NS]
  uint64_t* v_full = k_full + NS;   // [NS]
  uint64_t* k_pfull = v_full + NS;  // [NS] rank 0: rank 1's K half has landed
  uint64_t* v_pfull = k_pfull + NS; // [NS] rank 0: rank 1's V half has landed
  uint64_t* kv_empty = v_pfull + NS;
  uint64_t* q_empty = kv_empty + NS;
  uint64_t* s_full = q_empty + 1;   // [2]
  uint64_t* p_full = s_full + 2;    // [2] rank 0: both CTAs' P_t are in tensor memory
  uint64_t* o_done = p_full + 2;    // [2]
  uint64_t* o_free = o_done + 2;    // [2] rank 0: both CTAs' epilogues have read O_t
  uint64_t* drain = o_free + 2;
  uint64_t* exit_bar = drain + 1;   // the peer has finished with this CTA's memory
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const int G = (int)nclusters_x(), pc = (int)cluster_id_x();

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_pfull, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_pfull[s], 1);
      mbar_init(&v_pfull[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(q_empty, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 8);  // four softmax warps in each CTA
      mbar_init(&o_done[t], 1);
      mbar_init(&o_free[t], 8);
    }
    mbar_init(drain, 1);
    mbar_init(exit_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc_pair(tmem_holder, C::kTmemCols);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised, both allocations made
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t peer_tmem = ld_shared_cluster_u32(mapa_shared(smem_u32(tmem_holder), rank ^ 1));
  const bool pair_ok = peer_tmem == tmem;  // the same answer in both CTAs
  if (!pair_ok && threadIdx.x == 0 && rank == 0) record_timeout(kErrPairTmem);
  const uint64_t limit = p.wait_limit;
  auto leader = [&](uint64_t* bar) { return mapa_shared(smem_u32(bar), 0); };

  if (!pair_ok) {
    // no work: fall through to the exit handshake
  } else if (warp == 8 && p.stall) {
    // Failure tests: the producer withholds every copy; the consumers' waits run out.
  } else if (warp == 8) {
    // ------------------------------ TMA producer (both CTAs) ------------------------------
    if (elect_one()) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k64);
      tma_prefetch_map(&map_v);
    }
    __syncwarp();
    int q_loads = 0, kv_loads = 0;
    for (int k = 0;; ++k) {
      const int item = fwd_sched_item(sched, k, G, pc, n_items);
      if (item < 0) break;
      FwdPairItem it;
      if (!fwd_pair_item_geom<PACKED>(p, item, nsb_max, it)) continue;
      // Q of the previous item must have been read by all its S products (q_empty: one
      // multicast completion per item after its last S; the next one needs this copy).
      if (q_loads > 0 &&
          !warp_wait(q_empty, (q_loads - 1) & 1, limit, abort_flag, kWaitFwdQEmpty))
        break;
      const int ntiles = it.nkv[1] > 0 ? 2 : 1;
      if (elect_one()) {
        mbar_arrive_expect_tx(q_full, ntiles * C::kQTileBytes);
        for (int t = 0; t < ntiles; ++t)
          for (int c = 0; c < 2; ++c)
            tma_load_rows<PACKED>(smem + C::kOffQ + t * C::kQTileBytes + c * kBoxBytes, &map_q,
                                  q_full, c * kBoxCols,
                                  it.q0 + t * 2 * kTileM + (int)rank * kTileM, it.sl, false);
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
          // K_j rows [64r, 64r + 64): two 64-column chunks of 64 rows
          mbar_arrive_expect_tx(&k_full[s], C::kKHalfBytes);
          for (int c = 0; c < 2; ++c)
            tma_load_rows<PACKED>(smem + C::kOffK + s * C::kKHalfBytes + c * C::kKChunkBytes,
                                  &map_k64, &k_full[s], c * kBoxCols,
                                  j * kTileN + (int)rank * (kTileN / 2), it.sl, true);
          // V_j columns [64r, 64r + 64), all 128 keys
          mbar_arrive_expect_tx(&v_full[s], C::kVHalfBytes);
          tma_load_rows<PACKED>(smem + C::kOffV + s * C::kVHalfBytes, &map_v, &v_full[s],
                                (int)rank * kBoxCols, j * kTileN, it.sl, true);
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
  } else if (warp == 9 && rank == 1) {
    // ------------------------------ forwarder (rank 1) ------------------------------------
    // Rank 1's copies complete on its own barriers; rank 0 learns of each one here, in the
    // order the producer issued them.
    const uint32_t q_pf = leader(q_pfull);
    int q_fw = 0, kv_fw = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = fwd_sched_item(sched, k, G, pc, n_items);
      if (item < 0) break;
      FwdPairItem it;
      if (!fwd_pair_item_geom<PACKED>(p, item, nsb_max, it)) continue;
      if (!(ok = warp_wait(q_full, q_fw & 1, limit, abort_flag, kWaitFwdQ))) break;
      warp_arrive_cluster(q_pf);
      ++q_fw;
      for (int j = 0; ok && j < it.n_kv; ++j) {
        const int s = kv_fw % NS;
        if (!(ok = warp_wait(&k_full[s], (kv_fw / NS) & 1, limit, abort_flag, kWaitFwdK)))
          break;
        warp_arrive_cluster(leader(&k_pfull[s]));
        if (!(ok = warp_wait(&v_full[s], (kv_fw / NS) & 1, limit, abort_flag, kWaitFwdV)))
          break;
        warp_arrive_cluster(leader(&v_pfull[s]));
        ++kv_fw;
      }
    }
    // The pair's MMAs read this CTA's memory until rank 0's drain commit lands here.
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitFwdDrain);
  } else if (warp == 9) {
    // ------------------------------ MMA issuer (rank 0) -----------------------------------
    const uint32_t idesc_s = make_idesc(BF16, 256, kTileN, false, false);
    const uint32_t idesc_o = make_idesc(BF16, 256, D, false, true);
    const uint64_t dq0 = make_sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t dk0 = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dv0 = make_sdesc_sw128(smem_u32(smem + C::kOffV), kBoxBytes, 1024);
    const uint32_t col_s[2] = {C::kColS0, C::kColS1};
    const uint32_t col_o[2] = {C::kColO0, C::kColO1};
    auto issue_s = [&](int t, int stage) {
      // S_t (256 x 128) = Q_t K_j^T over d: Q_t K-major [128 rows x 128] in each CTA, K_j
      // K-major [64 keys x 128] in each CTA (chunks of 64 rows, 8 KiB apart).
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qa = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        const uint32_t kb = ((kk >> 2) * C::kKChunkBytes + (kk & 3) * 32) >> 4;
        mma_ss_pair(tmem + col_s[t], dq0 + ((t * C::kQTileBytes) >> 4) + qa,
                    dk0 + ((stage * C::kKHalfBytes) >> 4) + kb, idesc_s, kk > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int t, int stage, bool acc) {
      // O_t (256 x d) += P_t V_j: P_t from each CTA's tensor memory (16-bit pairs over S_t),
      // V_j MN-major [128 keys x 64 columns] in each CTA.
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        mma_ts_pair(tmem + col_o[t], tmem + col_s[t] + kk * 8,
                    dv0 + ((stage * C::kVHalfBytes + kk * 2048) >> 4), idesc_o,
                    (acc || kk > 0) ? 1u : 0u);
    };
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) mma_commit_pair(bar, kBoth);
      __syncwarp();
    };
    // both this CTA's copy and rank 1's (forwarded) of one stage
    auto wait_stage = [&](uint64_t* own, uint64_t* peer, uint32_t parity, int where) {
      return warp_wait(own, parity, limit, abort_flag, where) &&
             __all_sync(0xffffffffu,
                        mbar_poll_cluster(peer, parity, limit, abort_flag, kWaitFwdPeer));
    };
    auto wait_cl = [&](uint64_t* bar, uint32_t parity, int where) {
      return __all_sync(0xffffffffu, mbar_poll_cluster(bar, parity, limit, abort_flag, where));
    };
    int q_used = 0, kv_base = 0;
    int tb[2] = {0, 0}, ti[2] = {0, 0};
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = fwd_sched_item(sched, k, G, pc, n_items);
      if (item < 0) break;
      FwdPairItem it;
      if (!fwd_pair_item_geom<PACKED>(p, item, nsb_max, it)) continue;
      const int n_kv = it.n_kv;
      if (!(ok = wait_stage(q_full, q_pfull, q_used & 1, kWaitFwdQ))) break;
      ++q_used;
      if (!(ok = wait_stage(&k_full[kv_base % NS], &k_pfull[kv_base % NS],
                            (kv_base / NS) & 1, kWaitFwdK)))
        break;
      // First S of each tile: it overwrites S_t, whose last P was read by a P V that the
      // tensor core runs before this product.
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (it.nkv[t] == 0) continue;
        tc_fence_after();
        if (elect_one()) {
          issue_s(t, kv_base % NS);
          mma_commit_pair(&s_full[t], kBoth);
        }
        __syncwarp();
      }
      if (n_kv == 1) commit(q_empty);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int b = kv_base + j, bn = b + 1;
        const int s = b % NS, sn = bn % NS;
        const int jn = j + 1;
        if (!(ok = wait_stage(&v_full[s], &v_pfull[s], (b / NS) & 1, kWaitFwdV))) break;
        tc_fence_after();
        bool next_k_ready = false;
#pragma unroll
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= it.nkv[t]) continue;
          // The first P V of an item overwrites O_t: both epilogues of the tile's previous
          // item must have read it.
          if (j == 0 && ti[t] > 0 && !(ok = wait_cl(&o_free[t], (ti[t] - 1) & 1, kWaitFwdOFree)))
            break;
          if (!(ok = wait_cl(&p_full[t], (tb[t] + j) & 1, kWaitFwdP))) break;
          tc_fence_after();
          if (elect_one()) {
            issue_pv(t, s, j > 0);
            mma_commit_pair(&o_done[t], kBoth);
          }
          __syncwarp();
          if (jn < it.nkv[t]) {
            if (!next_k_ready) {
              if (!(ok = wait_stage(&k_full[sn], &k_pfull[sn], (bn / NS) & 1, kWaitFwdK)))
                break;
              tc_fence_after();
              next_k_ready = true;
            }
            if (elect_one()) {
              issue_s(t, sn);
              mma_commit_pair(&s_full[t], kBoth);
            }
            __syncwarp();
          }
        }
        if (ok && jn == n_kv - 1) commit(q_empty);
        if (ok) commit(&kv_empty[s]);
      }
      kv_base += n_kv;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        tb[t] += it.nkv[t];
        ti[t] += it.nkv[t] > 0 ? 1 : 0;
      }
    }
    // Every MMA issued must finish before either CTA releases memory it reads.
    commit(drain);
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitFwdDrain);
  } else {
    // ------------------------------ softmax (tile t, this CTA's rows) ---------------------
    const int t = warp >> 2;
    const int wq = warp & 3;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + (t == 0 ? C::kColS0 : C::kColS1);
    const uint32_t t_o = tmem + lane_base + (t == 0 ? C::kColO0 : C::kColO1);
    const uint32_t p_full_l = leader(&p_full[t]);
    const uint32_t o_free_l = leader(&o_free[t]);
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
    int tb = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = fwd_sched_item(sched, k, G, pc, n_items);
      if (item < 0) break;
      FwdPairItem it;
      if (!fwd_pair_item_geom<PACKED>(p, item, nsb_max, it)) continue;
      const int nkv = t == 0 ? it.nkv[0] : it.nkv[1];
      if (nkv == 0) continue;
      const int tile_row0 = it.q0 + t * 2 * kTileM + (int)rank * kTileM;
      const int row = tile_row0 + wq * 32 + lane;
      float m = -INFINITY, l = 0.f, lr = 0.f;
      for (int j = 0; j < nkv; ++j) {
        const int b = tb + j;
        if (!(ok = warp_wait(&s_full[t], b & 1, limit, abort_flag, kWaitFwdS))) break;
        tc_fence_after();
        uint32_t sr[kTileN];
        tmem_ld128(t_s, sr);
        float* sv = reinterpret_cast<float*>(sr);
        const int kbase = j * kTileN;
        const bool diag = p.causal && (kbase + kTileN - 1 > tile_row0 + it.off);
        if (diag || kbase + kTileN > it.Nk) {
          int lim = it.Nk - 1 - kbase;
          if (p.causal) lim = min(lim, row + it.off - kbase);
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
          alpha = ex2(m - m_cand);
          m = m_cand;
        }
        const float2 sl2x2 = make_float2(sl2, sl2);
        const float2 neg_m2 = make_float2(-m, -m);
        float2 sum[4];
        float rsum[4] = {0.f, 0.f, 0.f, 0.f};
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
          tmem_st16(t_s + c4 * 16, pk);
        }
        const float2 sa = add2(add2(sum[0], sum[1]), add2(sum[2], sum[3]));
        l = l * alpha + (sa.x + sa.y);
        lr = lr * alpha + ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3]));
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          if (!(ok = warp_wait(&o_done[t], (b - 1) & 1, limit, abort_flag, kWaitFwdO))) break;
          tc_fence_after();
          rescale_o(alpha);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive_cluster(p_full_l);
      }
      if (!ok) break;
      if (!(ok = warp_wait(&o_done[t], (tb + nkv - 1) & 1, limit, abort_flag, kWaitFwdO)))
        break;
      tc_fence_after();
      uint32_t r[D];
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc)
        tmem_ld64(t_o + cc * 64, *reinterpret_cast<uint32_t(*)[64]>(&r[cc * 64]));
      tc_fence_before();
      warp_arrive_cluster(o_free_l);
      tb += nkv;
      if (row < it.N) {
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
          const int n16 = valid16(p.dh, cc * 64, 8);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            if (v < n16)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
        p.lse[it.sl.stat0 + row] = (m + log2f(l)) * kLn2;
      }
    }
    tc_fence_before();
  }

  // ------------------------------ exit handshake ------------------------------------------
  tmem_st_wait();  // no tensor-memory store in flight
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_cluster(mapa_shared(smem_u32(exit_bar), rank ^ 1));
    mbar_wait_cluster(exit_bar, 0, kDrainLimit, nullptr, kWaitFwdExit);
  }
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

}  // namespace attn
