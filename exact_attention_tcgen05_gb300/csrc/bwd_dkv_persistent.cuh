// bwd_dkv_persistent.cuh - the dK/dV kernel of bwd_dkv.cuh as a persistent kernel: one CTA
// per SM walks a list of work items (128 keys of one (b, h) slice each), for short items.
//
// Why: a CTA of the one-item kernel pays a fixed cost of about 5-7 us (launch, set-up, the
// K_j/V_j copy, the pipeline's first query block, the dK/dV epilogue), measured on GB300 by
// timing whole waves of CTAs; with few query blocks per key block (short or causal
// sequences) that is about half of the kernel's time. Here the Q/dO ring, the barrier
// phases and the tensor memory carry over from one item to the next: the next item's K_j
// and V_j are copied as soon as the current item's last S^T and dP^T products have read
// the current ones, and its first products run while the current item's dK/dV are written.
//
// The arithmetic of every item is exactly that of bwd_dkv.cuh (K_j, V_j in shared memory):
// the outputs are bit-identical.
//
// Schedule: as for the persistent dQ kernel - a greedy table (schedule.h) for dense causal
// inputs with more items than CTAs, otherwise key block p of a slice paired with block
// nkb - 1 - p (a long and a short causal block) and the pairs dealt round-robin.
#pragma once

#include "bwd_dkv.cuh"
#include "bwd_dq_persistent.cuh"

namespace attn {

// One dK/dV work item.
struct DkvItem {
  SliceRows sl;
  int N, Nk, off;
  int j0;       // first key of the block
  int i_first;  // first query block that sees it
  int n;        // query blocks i_first .. i_first + n - 1; 0: a packed sequence without
                // queries, whose key gradients are zero
};

// Geometry of dK/dV item `item` (nkb_max key blocks per slice). False: nothing to do.
template <int D, bool PACKED>
__device__ __forceinline__ bool dkv_item_geom(const BwdParams& p, int item, int nkb_max,
                                              DkvItem& it) {
  const int bh = item / nkb_max;
  const int jb = item - bh * nkb_max;  // jb = 0: the longest causal block
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, it.sl)) return false;
  it.N = it.sl.nq;
  it.Nk = it.sl.nk;
  it.off = it.sl.off;
  if (jb * kTileN >= it.Nk) return false;
  it.j0 = jb * kTileN;
  const int nb = (it.N + kTileM - 1) / kTileM;
  it.i_first = (p.causal && it.j0 > it.off) ? (it.j0 - it.off) / kTileM : 0;
  it.n = it.N == 0 ? 0 : nb - it.i_first;
  return true;
}

template <int D>
struct DkvPCfg : DkvCfg<D> {
  using B = DkvCfg<D>;
  // Q and dO in rings of their own depths. A Q block's last reader is dK += dS^T Q, a dO
  // block's dV += P^T dO, which the tensor core runs earlier; so at d = 128, where the
  // Q + dO copies of a block barely keep up with its work, Q gets three slots and dO two
  // (with K_j, V_j: 224 KiB of tiles; measured on GB300 against two of each: B4 H32 N4096
// dK/dV 0.781 -> 0.757 ms). d = 64: three of each.
  static constexpr int kQStages = D == 128 ? 3 : B::kStages;
  static constexpr int kDOStages = B::kStages;
  static constexpr int kOffQ = B::kOffQ;  // after K_j, V_j
  static constexpr int kOffDO = kOffQ + kQStages * B::kTileBytes;
  static constexpr int kOffStats = kOffDO + kDOStages * B::kTileBytes;
  static constexpr int kOffBar = kOffStats + 2 * 256 * 4;
  // kv_full, q_full[QS], do_full[DS], q_empty[QS], do_empty[DS], s_full, p_full, dp_full,
  // ds_full, acc_done, drain, stats_ready[2], kv_free, acc_free
  static constexpr int kNumBars = 1 + 2 * kQStages + 2 * kDOStages + 8 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // d = 64: each elementwise warp stages its 32 rows of dV or dK in shared memory (4 KiB,
  // 128-byte swizzle) and writes them with one TMA store, instead of 16-byte stores row by
  // row (dense tensors; packed batches keep the row stores, since a key block may run past
  // its sequence into the next one's rows).
  static constexpr bool kStageOut = (D == 64);
  static constexpr int kOffOut = ((kOffMisc + 16 + 1023) / 1024) * 1024;
  static constexpr int kEnd = kStageOut ? kOffOut + 8 * 4096 : kOffMisc + 16;
  // 1024 bytes of slack to align the dynamic shared memory's base, where they fit in the
  // 227 KiB a CTA may take; otherwise none, and the kernel checks that the base is aligned
  // (it is on GB300: no static shared memory comes before it).
  static constexpr int kLimit = 227 * 1024;
  static constexpr int kSlack = (kEnd + 1024 <= kLimit) ? 1024 : 0;
  static constexpr int kSmemBytes = (kEnd + kSlack) > B::kMinSmem ? (kEnd + kSlack) : B::kMinSmem;
  static_assert(kSmemBytes <= kLimit, "shared memory");
  static_assert(!kStageOut || kSlack == 1024, "the staging buffers need an aligned base");
};

template <int D, bool BF16, bool PACKED, class Sched>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_dkv_persistent_kernel(const __grid_constant__ CUtensorMap map_q,
                                   const __grid_constant__ CUtensorMap map_k,
                                   const __grid_constant__ CUtensorMap map_v,
                                   const __grid_constant__ CUtensorMap map_do,
                                   const __grid_constant__ CUtensorMap map_dk,
                                   const __grid_constant__ CUtensorMap map_dv,
                                   const BwdParams p, int n_pairs, int npairs, int nkb_max,
                                   const __grid_constant__ Sched sched) {
  using C = DkvPCfg<D>;
  constexpr bool kTmaOut = C::kStageOut && !PACKED;
  constexpr int QS = C::kQStages, DS = C::kDOStages;
  // Rings of different depths release their slots separately (dO after the block's dV
  // product, Q after its dK product); at equal depths one release per block covers both
  // (q_empty, committed after the block's last product), which measured 1% faster at d = 64.
  constexpr bool kSplit = QS != DS;
  extern __shared__ uint8_t smem_raw[];
  if (C::kSlack == 0 && (smem_u32(smem_raw) & 1023u) != 0) {
    // Without slack the layout needs an aligned base: report and do nothing (every thread
    // takes this branch, before any barrier or tensor memory is set up).
    if (threadIdx.x == 0) record_timeout(kErrSmemAlign);
    return;
  }
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;          // [QS]
  uint64_t* do_full = q_full + QS;      // [DS]
  uint64_t* q_empty = do_full + DS;     // [QS] the block's dK product has read Q_i
  uint64_t* do_empty = q_empty + QS;    // [DS] the block's dV product has read dO_i
  uint64_t* s_full = do_empty + DS;
  uint64_t* p_full = s_full + 1;
  uint64_t* dp_full = p_full + 1;
  uint64_t* ds_full = dp_full + 1;
  uint64_t* acc_done = ds_full + 1;
  uint64_t* drain = acc_done + 1;
  uint64_t* stats_ready = drain + 1;  // [2], one per statistics buffer
  uint64_t* kv_free = stats_ready + 2;  // the item's S^T, dP^T have read K_j, V_j
  uint64_t* acc_free = kv_free + 1;  // the epilogue has read dK, dV
  float* stats = reinterpret_cast<float*>(smem + C::kOffStats);  // [2][-L*log2e x128, D x128]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < QS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < DS; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 8);  // one arrival per elementwise warp
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 8);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    mbar_init(&stats_ready[0], 8);
    mbar_init(&stats_ready[1], 8);
    mbar_init(kv_free, 1);
    mbar_init(acc_free, 8);
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
    // TMA producer: K_j, V_j per item, and the Q/dO ring continued across items.
    if (elect_one()) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      tma_prefetch_map(&map_do);
    }
    __syncwarp();
    int kv_loads = 0, q_loads = 0, do_loads = 0;  // K/V (items), Q and dO copies so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = sched_item(sched, k, G, cta, n_pairs, npairs, nkb_max);
      if (item == -1) break;
      DkvItem it;
      if (item < 0 || !dkv_item_geom<D, PACKED>(p, item, nkb_max, it) || it.n == 0) continue;
      // K_j, V_j of the previous item must have been read by all its S^T and dP^T products
      // (kv_free: one commit per item after its last dP^T; the next needs this copy).
      if (kv_loads > 0 &&
          !(ok = warp_wait(kv_free, (kv_loads - 1) & 1, limit, abort_flag, kWaitDkvKVFree)))
        break;
      if (elect_one()) {
        mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_rows<PACKED>(smem + C::kOffK + c * kBoxBytes, &map_k, kv_full,
                                c * kBoxCols, it.j0, it.sl, true);
          tma_load_rows<PACKED>(smem + C::kOffV + c * kBoxBytes, &map_v, kv_full,
                                c * kBoxCols, it.j0, it.sl, true);
        }
      }
      __syncwarp();
      ++kv_loads;
      for (int t = 0; t < it.n; ++t) {
        const int i = it.i_first + t;
        // Q_i into its slot once the block that held it has had its dK product (q_empty:
        // one completion per block using the slot; the next needs this copy), dO_i once
        // its slot's block has had its dV product. Waited in the order the slots free up:
        // Q first when its ring is deeper (dK of block b - QS runs before dV of block
        // b - DS), dO first at equal depths (dV runs before dK of the same block).
        auto load_q = [&]() -> bool {
          const int sq = q_loads % QS;
          if (q_loads >= QS && !warp_wait(&q_empty[sq], ((q_loads / QS) - 1) & 1, limit,
                                          abort_flag, kWaitDkvEmpty))
            return false;
          if (elect_one()) {
            mbar_arrive_expect_tx(&q_full[sq], C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_rows<PACKED>(smem + C::kOffQ + sq * C::kTileBytes + c * kBoxBytes,
                                    &map_q, &q_full[sq], c * kBoxCols, i * kTileM, it.sl,
                                    false);
          }
          __syncwarp();
          ++q_loads;
          return true;
        };
        auto load_do = [&]() -> bool {
          const int sd = do_loads % DS;
          if (do_loads >= DS && !warp_wait(&do_empty[sd], ((do_loads / DS) - 1) & 1, limit,
                                           abort_flag, kWaitDkvEmpty))
            return false;
          if (elect_one()) {
            mbar_arrive_expect_tx(&do_full[sd], C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_rows<PACKED>(smem + C::kOffDO + sd * C::kTileBytes + c * kBoxBytes,
                                    &map_do, &do_full[sd], c * kBoxCols, i * kTileM, it.sl,
                                    false);
          }
          __syncwarp();
          ++do_loads;
          return true;
        };
        if constexpr (!kSplit) {
          // one slot index for both rings: q_empty is the block's combined release
          const int s = q_loads % QS;
          if (q_loads >= QS && !(ok = warp_wait(&q_empty[s], ((q_loads / QS) - 1) & 1, limit,
                                                abort_flag, kWaitDkvEmpty)))
            break;
          if (elect_one()) {
            mbar_arrive_expect_tx(&q_full[s], C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_rows<PACKED>(smem + C::kOffQ + s * C::kTileBytes + c * kBoxBytes,
                                    &map_q, &q_full[s], c * kBoxCols, i * kTileM, it.sl,
                                    false);
            mbar_arrive_expect_tx(&do_full[s], C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_rows<PACKED>(smem + C::kOffDO + s * C::kTileBytes + c * kBoxBytes,
                                    &map_do, &do_full[s], c * kBoxCols, i * kTileM, it.sl,
                                    false);
          }
          __syncwarp();
          ++q_loads;
          ++do_loads;
        } else {
          if (QS > DS)
            ok = load_q() && load_do();
          else
            ok = load_do() && load_q();
          if (!ok) break;
        }
      }
    }
    if (*abort_flag) {
      if (kv_loads > 0)
        mbar_wait(kv_full, (kv_loads - 1) & 1, kDrainLimit, nullptr, kWaitDkvDrain);
      for (int b = max(0, q_loads - QS); b < q_loads; ++b)
        mbar_wait(&q_full[b % QS], (b / QS) & 1, kDrainLimit, nullptr, kWaitDkvDrain);
      for (int b = max(0, do_loads - DS); b < do_loads; ++b)
        mbar_wait(&do_full[b % DS], (b / DS) & 1, kDrainLimit, nullptr, kWaitDkvDrain);
    }
  }
  else if (warp == 9) {
    // MMA issuer (converged warp, elected lane issues), as in bwd_dkv.cuh, with the block
    // count b running across items.
    const uint32_t idesc_st = make_idesc(BF16, 128, kTileM, false, false);
    const uint32_t idesc_acc = make_idesc(BF16, 128, D, false, true);
    const uint64_t dk = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dv = make_sdesc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
    const uint64_t dq = make_sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t ddo = make_sdesc_sw128(smem_u32(smem + C::kOffDO), 16, 1024);
    const uint64_t dq_mn = make_sdesc_sw128(smem_u32(smem + C::kOffQ), kBoxBytes, 1024);
    const uint64_t ddo_mn = make_sdesc_sw128(smem_u32(smem + C::kOffDO), kBoxBytes, 1024);
    constexpr uint32_t kStageStep = C::kTileBytes >> 4;
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) mma_commit(bar);
      __syncwarp();
    };
    int items = 0, tb = 0;  // items and blocks so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = sched_item(sched, k, G, cta, n_pairs, npairs, nkb_max);
      if (item == -1) break;
      DkvItem it;
      if (item < 0 || !dkv_item_geom<D, PACKED>(p, item, nkb_max, it) || it.n == 0) continue;
      const int n = it.n;
      // K_j, V_j of this item (kv_full: one completion per item; the next copy needs the
      // kv_free committed below) and its first Q block.
      if (!(ok = warp_wait(kv_full, items & 1, limit, abort_flag, kWaitDkvKV) &&
                 warp_wait(&q_full[tb % QS], (tb / QS) & 1, limit, abort_flag, kWaitDkvQ)))
        break;
      // S^T overwrites the previous item's last P^T, read by a dV product the tensor core
      // runs before this one; dP^T likewise the last dS^T, read by the last dK product.
      tc_fence_after();
      if (elect_one()) {
        issue_rowdot_d<D>(tmem + C::kColS, dk, dq + (tb % QS) * kStageStep, idesc_st);
        mma_commit(s_full);
      }
      __syncwarp();
      if (!(ok = warp_wait(&do_full[tb % DS], (tb / DS) & 1, limit, abort_flag, kWaitDkvDO)))
        break;
      tc_fence_after();
      if (elect_one()) {
        issue_rowdot_d<D>(tmem + C::kColDP, dv, ddo + (tb % DS) * kStageStep, idesc_st);
        mma_commit(dp_full);
      }
      __syncwarp();
      if (n == 1) commit(kv_free);  // every S^T and dP^T of the item issued
      for (int t = 0; ok && t < n; ++t) {
        const int b = tb + t, bn = b + 1;
        const int sq = b % QS, sqn = bn % QS, sd = b % DS, sdn = bn % DS;
        if (!(ok = warp_wait(p_full, b & 1, limit, abort_flag, kWaitDkvP))) break;
        // The first accumulating products of an item overwrite dV and dK: the previous
        // item's epilogue must have read them (acc_free: one completion per item, each
        // after an acc_done that follows this wait).
        if (t == 0 && items > 0 &&
            !(ok = warp_wait(acc_free, (items - 1) & 1, limit, abort_flag, kWaitDkvAccFree)))
          break;
        tc_fence_after();
        // dV_j += P^T dO_i, the last reader of dO_i's slot
        if (elect_one())
          issue_tmem_a_split_d(tmem + C::kColAcc0, tmem + C::kColS, ddo_mn + sd * kStageStep,
                               idesc_acc, t > 0);
        __syncwarp();
        if constexpr (kSplit) commit(&do_empty[sd]);
        if (t + 1 < n) {
          if (!(ok = warp_wait(&q_full[sqn], (bn / QS) & 1, limit, abort_flag, kWaitDkvQ)))
            break;
          tc_fence_after();
          if (elect_one()) {
            issue_rowdot_d<D>(tmem + C::kColS, dk, dq + sqn * kStageStep, idesc_st);
            mma_commit(s_full);
          }
          __syncwarp();
        }
        if (!(ok = warp_wait(ds_full, b & 1, limit, abort_flag, kWaitDkvDS))) break;
        tc_fence_after();
        // dK_j += dS^T Q_i, the last reader of Q_i's slot
        if (elect_one())
          issue_tmem_a_split_d(tmem + C::kColAcc1, tmem + C::kColDP, dq_mn + sq * kStageStep,
                               idesc_acc, t > 0);
        __syncwarp();
        if constexpr (kSplit) commit(&q_empty[sq]);
        if (t + 1 < n) {
          if (!(ok = warp_wait(&do_full[sdn], (bn / DS) & 1, limit, abort_flag, kWaitDkvDO)))
            break;
          tc_fence_after();
          if (elect_one()) {
            issue_rowdot_d<D>(tmem + C::kColDP, dv, ddo + sdn * kStageStep, idesc_st);
            mma_commit(dp_full);
          }
          __syncwarp();
          if (t + 2 == n) commit(kv_free);
        }
        if constexpr (!kSplit) commit(&q_empty[sq]);  // both slots of block b
      }
      if (!ok) break;
      commit(acc_done);
      tb += n;
      ++items;
    }
    commit(drain);
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitDkvDrain);
  }
  else {
    // warps 0-7: thread = key row (TMEM lane); group g covers queries [64g, 64g + 64)
    const int g = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // 0..127
    const int c0 = g * 64;           // first query column of this group
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::kColS + c0;
    const uint32_t t_dp = tmem + lane_base + C::kColDP + c0;
    const float2 sl2x2 = make_float2(p.scale_log2, p.scale_log2);
    int items = 0, tb = 0;  // items and blocks so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = sched_item(sched, k, G, cta, n_pairs, npairs, nkb_max);
      if (item == -1) break;
      DkvItem it;
      if (item < 0 || !dkv_item_geom<D, PACKED>(p, item, nkb_max, it)) continue;
      const int key = it.j0 + row;
      if (it.n == 0) {
        // A packed sequence with keys but no queries: their gradients are zero.
        if (key < it.Nk) {
          for (int t = 0; t < 2; ++t) {
            uint8_t* base = reinterpret_cast<uint8_t*>(t == 0 ? p.out0 : p.out1);
            uint4* dst = reinterpret_cast<uint4*>(
                base + (it.sl.k_elem0 + (size_t)key * it.sl.row_elems) * 2);
            for (int c = g; c < p.dh / 8; c += 2) dst[c] = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      // Group 0 stages -L*log2(e), group 1 stages D: one value per thread per query block.
      const float* src = (g == 0 ? p.lse : p.delta) + it.sl.stat0;
      auto load_stat = [&](int i) -> float {
        const int q = i * kTileM + row;
        if (q >= it.N) return g == 0 ? -INFINITY : 0.f;  // padding queries: P = 0, D = 0
        const float x = src[q];
        return g == 0 ? -x * kLog2e : x;
      };
      float stat_next = load_stat(it.i_first);
      for (int t = 0; t < it.n; ++t) {
        const int b = tb + t;
        const int i = it.i_first + t;
        // Double-buffered statistics (running block count): buffer b&1 was last read in
        // block b-2, and every thread has passed block b-1's stats_ready wait.
        float* st = stats + (b & 1) * 256;
        st[g * 128 + row] = stat_next;
        warp_arrive(&stats_ready[b & 1]);
        if (t + 1 < it.n) stat_next = load_stat(i + 1);
        if (!(ok = warp_wait(&stats_ready[b & 1], (b >> 1) & 1, limit, abort_flag,
                             kWaitDkvStats)))
          break;
        // ---- P^T = exp2(S^T * scale * log2(e) - L * log2(e)), 16-bit pairs over S^T
        if (!(ok = warp_wait(s_full, b & 1, limit, abort_flag, kWaitDkvS))) break;
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64(t_s, sr);
        float* pr = reinterpret_cast<float*>(sr);
        const float4* nl4 = reinterpret_cast<const float4*>(st + c0);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 nl = nl4[c4];
          const float2 a = fma2(make_float2(pr[4 * c4], pr[4 * c4 + 1]), sl2x2,
                                make_float2(nl.x, nl.y));
          const float2 bb = fma2(make_float2(pr[4 * c4 + 2], pr[4 * c4 + 3]), sl2x2,
                                 make_float2(nl.z, nl.w));
          pr[4 * c4] = ex2(a.x);
          pr[4 * c4 + 1] = ex2(a.y);
          pr[4 * c4 + 2] = ex2(bb.x);
          pr[4 * c4 + 3] = ex2(bb.y);
        }
        if (p.causal && i * kTileM + it.off < it.j0 + kTileN - 1) {
          // A block on the diagonal: query i*128 + c0 + c sees this key iff
          // i*128 + c0 + c + off >= key, i.e. c >= key - off - i*128 - c0.
          const int first = key - it.off - i * kTileM - c0;
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < first) pr[c] = 0.f;
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) pk[u] = pack2<BF16>(pr[2 * u], pr[2 * u + 1]);
          uint32_t (&lo)[16] = *reinterpret_cast<uint32_t(*)[16]>(&pk[0]);
          uint32_t (&hi)[16] = *reinterpret_cast<uint32_t(*)[16]>(&pk[16]);
          tmem_st16(t_s, lo);
          tmem_st16(t_s + 16, hi);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(p_full);
        // ---- dS^T = P^T * (dP^T - D), 16-bit pairs over dP^T
        if (!(ok = warp_wait(dp_full, b & 1, limit, abort_flag, kWaitDkvDP))) break;
        tc_fence_after();
        uint32_t r[64];
        tmem_ld64(t_dp, r);
        const float4* dl4 = reinterpret_cast<const float4*>(st + 128 + c0);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float4 dl = dl4[u];
          const float2 d01 = mul2(make_float2(pr[4 * u], pr[4 * u + 1]),
                                  add2(make_float2(__uint_as_float(r[4 * u]),
                                                   __uint_as_float(r[4 * u + 1])),
                                       make_float2(-dl.x, -dl.y)));
          const float2 d23 = mul2(make_float2(pr[4 * u + 2], pr[4 * u + 3]),
                                  add2(make_float2(__uint_as_float(r[4 * u + 2]),
                                                   __uint_as_float(r[4 * u + 3])),
                                       make_float2(-dl.z, -dl.w)));
          r[2 * u] = pack2<BF16>(d01.x, d01.y);
          r[2 * u + 1] = pack2<BF16>(d23.x, d23.y);
        }
        {
          uint32_t (&lo)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[0]);
          uint32_t (&hi)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[16]);
          tmem_st16(t_dp, lo);
          tmem_st16(t_dp + 16, hi);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(ds_full);
      }
      if (!ok) break;
      tb += it.n;
      // Epilogue: group 0 writes dV, group 1 dK (scaled); then the accumulators are free
      // for the next item's first products (acc_free).
      if (!(ok = warp_wait(acc_done, items & 1, limit, abort_flag, kWaitDkvDone))) break;
      tc_fence_after();
      const uint32_t t_acc = tmem + lane_base + (g == 0 ? C::kColAcc0 : C::kColAcc1);
      const float mul = (g == 0) ? 1.f : p.scale;
      if constexpr (kTmaOut) {
        // All of the row into registers, the accumulators released at once (the next
        // item's first products may overwrite them), then the row staged in this warp's
        // buffer and the warp's 32 rows stored by one TMA copy once the buffer's previous
        // store has read it.
        uint32_t a[D];
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc)
          tmem_ld32(t_acc + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&a[cc * 32]));
        tc_fence_before();
        warp_arrive(acc_free);
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        uint8_t* buf = smem + C::kOffOut + warp * 4096;
        const uint32_t rbase = smem_u32(buf) + lane * 128;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint32_t w4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            w4[i] = pack2<BF16>(__uint_as_float(a[8 * v + 2 * i]) * mul,
                                __uint_as_float(a[8 * v + 2 * i + 1]) * mul);
          st_shared_v4(rbase + ((v ^ (lane & 7)) << 4), w4[0], w4[1], w4[2], w4[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(g == 0 ? &map_dv : &map_dk, buf, 0, it.j0 + wq * 32, it.sl.tma_bh);
          bulk_commit_group();
        }
      } else {
        uint8_t* dst = reinterpret_cast<uint8_t*>(g == 0 ? p.out1 : p.out0) +
                       (it.sl.k_elem0 + (size_t)key * it.sl.row_elems) * 2;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t a[32];
          tmem_ld32(t_acc + cc * 32, a);
          if (key < it.Nk) store_row32<BF16>(dst + cc * 64, a, mul, valid16(p.dh, cc * 32, 4));
        }
        tc_fence_before();
        warp_arrive(acc_free);
      }
      ++items;
    }
    // the warp's last store must have finished with its buffer before shared memory is
    // released
    if (kTmaOut && lane == 0) bulk_wait_all();
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
