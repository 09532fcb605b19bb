// bwd_dq_persistent.cuh - the dQ kernel of bwd_dq.cuh as a persistent kernel: one CTA per
// SM walks a list of work items (128 query rows of one (b, h) slice each).
//
// Why: a CTA of the one-item kernel pays a fixed cost of about 7 us at d = 128 (launch,
// set-up, the copy of its Q_i and dO_i rows into tensor memory, the pipeline's first
// block, the dQ epilogue), measured on GB300 by timing whole waves of CTAs with 1 to 16
// key blocks each - as much as eight key blocks of work. Here the pipeline keeps running
// from one item to the next: after the last dS of an item the elementwise warps load the
// next item's Q/dO rows and L/D, place them in tensor memory as soon as the last S and dP
// products have read the old ones, and only then write the finished dQ, so the tensor core
// starts on the next item while the epilogue runs. At d = 64 those rows are requested
// earlier, at the start of the item's last block, into shared memory (cp.async), so their
// latency hides behind that block (GPT-2-medium shape on GB300: 0.363 -> 0.341 ms).
//
// The arithmetic of every item is exactly that of bwd_dq.cuh: the outputs are
// bit-identical.
//
// Schedule (the kernel's Sched parameter): for dense causal inputs with more items than
// CTAs, a longest-first greedy table built on the host (schedule.h); otherwise the items of
// a slice are paired, query block p with block nb - 1 - p (a long and a short causal
// block: every pair carries the same work), and the pairs, numbered slice by slice, are
// dealt round-robin to the G CTAs. Either way the CTAs working at one time share the K/V
// of a few slices in L2.
//
// Barrier phases follow running counts kept alike by all roles (blocks, items); each
// barrier's next completion needs a step its waiter takes after the previous wait, so no
// wait can see a phase two ahead (the argument is at each new barrier below).
#pragma once

#include "bwd_dq.cuh"
#include "schedule.h"

namespace attn {

// One dQ work item.
struct DqItem {
  SliceRows sl;
  int N, Nk, off;
  int i0;  // first query row within the slice
  int n;   // key blocks 0 .. n-1
};

// The k-th item of CTA c among G: pair c + (k / 2) G, first or second half. -1: past the
// end; -2: nothing in this slot (the middle block of an odd count has no partner).
__device__ __forceinline__ int bwd_pair_item(int k, int G, int c, int n_pairs, int npairs,
                                             int nb_max) {
  const int pi = c + (k >> 1) * G;
  if (pi >= n_pairs) return -1;
  const int slice = pi / npairs, pp = pi - slice * npairs;
  const int x = (k & 1) ? nb_max - 1 - pp : pp;
  if ((k & 1) && x == pp) return -2;
  return slice * nb_max + x;
}

// The schedule types the persistent backward kernels take (by value, as a kernel
// parameter): the long/short pairs dealt round-robin above, or an ItemTable (schedule.h),
// which the host builds for dense causal inputs.
struct PairSchedule {};
__device__ __forceinline__ int sched_item(const PairSchedule&, int k, int G, int c, int n_pairs,
                                          int npairs, int nb_max) {
  return bwd_pair_item(k, G, c, n_pairs, npairs, nb_max);
}
__device__ __forceinline__ int sched_item(const ItemTable& t, int k, int, int c, int, int, int) {
  return table_item(t, k, c);
}

// Geometry of dQ item `item` (nb_max query blocks per slice). False: nothing to do.
template <int D, bool PACKED>
__device__ __forceinline__ bool dq_item_geom(const BwdParams& p, int item, int nb_max,
                                             DqItem& it) {
  const int bh = item / nb_max;
  const int x = item - bh * nb_max;
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, it.sl)) return false;
  it.N = it.sl.nq;
  it.Nk = it.sl.nk;
  it.off = it.sl.off;
  const int nb = (it.N + kTileM - 1) / kTileM;
  if (x >= nb) return false;
  const int nkb = (it.Nk + kTileN - 1) / kTileN;
  const int ib = p.causal ? (nb - 1 - x) : x;  // x = 0: the longest causal block
  it.i0 = ib * kTileM;
  it.n = p.causal ? min(nkb, (it.i0 + kTileM - 1 + it.off) / kTileN + 1) : nkb;
  return true;
}

template <int D>
struct DqPCfg : DqCfg<D> {
  using B = DqCfg<D>;
  // The barriers of the one-item kernel, then qdo_free and acc_free.
  static constexpr int kNumBars = B::kNumBars + 2;
  static constexpr int kOffMisc = B::kOffBar + kNumBars * 8;
  // d = 64: the next item's Q_i / dO_i rows are staged in shared memory (one 128-byte row
  // per elementwise thread, 32 KiB) while the current item's last block runs. At d = 128
  // the K/V ring leaves no room for the 64 KiB this would take.
  static constexpr bool kStageRows = D == 64;
  static constexpr int kOffStage = (kOffMisc + 16 + 127) / 128 * 128;
  static constexpr int kStageBytes = kStageRows ? 256 * (D * 2 + 8) : 0;
  // d = 64: each elementwise warp stages its 32 rows x 32 columns of dQ (64-byte rows,
  // unswizzled, 2 KiB) and writes them with one TMA store, instead of 16-byte stores row
  // by row (dense tensors; packed batches keep the row stores).
  static constexpr bool kStageOut = D == 64;
  static constexpr int kOffOut = (kOffStage + kStageBytes + 1023) / 1024 * 1024;
  static constexpr int kEnd = (kStageOut ? kOffOut + 8 * 2048 : kOffStage + kStageBytes) + 1024;
  static constexpr int kSmemBytes = kEnd > B::kMinSmem ? kEnd : B::kMinSmem;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// A D-element 16-bit row from global memory into registers as packed pairs (zeros when
// src is null), and those registers into tensor-memory columns [t_col, t_col + D/2) of
// this thread's lane: copy_row_to_tmem in two halves, so that the loads can be issued
// well before the tensor memory they go to is free.
template <int D>
__device__ __forceinline__ void load_row(const uint8_t* src, uint32_t (&r)[D / 2], int n16) {
#pragma unroll
  for (int k = 0; k < D / 8; ++k) {
    const uint4 v = (src && k < n16) ? *reinterpret_cast<const uint4*>(src + k * 16)
                                     : make_uint4(0, 0, 0, 0);
    r[4 * k] = v.x;
    r[4 * k + 1] = v.y;
    r[4 * k + 2] = v.z;
    r[4 * k + 3] = v.w;
  }
}
template <int D>
__device__ __forceinline__ void store_row_tmem(const uint32_t (&r)[D / 2], uint32_t t_col) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c)
    tmem_st32(t_col + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&r[32 * c]));
}

template <int D, bool BF16, bool PACKED, class Sched>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_dq_persistent_kernel(const __grid_constant__ CUtensorMap map_q,
                                  const __grid_constant__ CUtensorMap map_k,
                                  const __grid_constant__ CUtensorMap map_v,
                                  const __grid_constant__ CUtensorMap map_do,
                                  const __grid_constant__ CUtensorMap map_dq, const BwdParams p,
                                  int n_pairs, int npairs, int nb_max,
                                  const __grid_constant__ Sched sched) {
  using C = DqPCfg<D>;
  constexpr bool kTmaOut = C::kStageOut && !PACKED;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* k_full = bars;
  uint64_t* v_full = k_full + NS;
  uint64_t* kv_empty = v_full + NS;
  uint64_t* s_full = kv_empty + NS;
  uint64_t* s_free = s_full + 1;
  uint64_t* dp_full = s_free + 1;
  uint64_t* ds_full = dp_full + 1;
  uint64_t* acc_done = ds_full + 1;
  uint64_t* drain = acc_done + 1;
  uint64_t* qdo_tmem = drain + 1;  // the item's Q_i and dO_i rows are in tensor memory
  uint64_t* qdo_free = qdo_tmem + 1;  // the item's S and dP products have read them
  uint64_t* acc_free = qdo_free + 1;  // the epilogue has read the dQ accumulator
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 8);  // one arrival per elementwise warp
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 8);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    mbar_init(qdo_tmem, 8);
    mbar_init(qdo_free, 1);
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
    // TMA producer: the K/V ring, continued across items.
    if (elect_one()) {
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
    }
    __syncwarp();
    int loads = 0;  // ring blocks issued so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = sched_item(sched, k, G, cta, n_pairs, npairs, nb_max);
      if (item == -1) break;
      DqItem it;
      if (item < 0 || !dq_item_geom<D, PACKED>(p, item, nb_max, it)) continue;
      for (int j = 0; j < it.n; ++j) {
        const int s = loads % NS;
        if (loads >= NS &&
            !(ok = warp_wait(&kv_empty[s], ((loads / NS) - 1) & 1, limit, abort_flag,
                             kWaitDqEmpty)))
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
        ++loads;
      }
    }
    if (*abort_flag) {
      for (int b = max(0, loads - NS); b < loads; ++b) {
        mbar_wait(&k_full[b % NS], (b / NS) & 1, kDrainLimit, nullptr, kWaitDqDrain);
        mbar_wait(&v_full[b % NS], (b / NS) & 1, kDrainLimit, nullptr, kWaitDqDrain);
      }
    }
  }
  else if (warp == 9) {
    // MMA issuer (converged warp, elected lane issues), as in bwd_dq.cuh, with the block
    // count b running across items.
    const uint32_t idesc_sq = make_idesc(BF16, 128, kTileN, false, false);
    const uint32_t idesc_acc = make_idesc(BF16, 128, D, false, true);
    const uint64_t dk = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dk_mn = make_sdesc_sw128(smem_u32(smem + C::kOffK), kBoxBytes, 1024);
    const uint64_t dv = make_sdesc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
    constexpr uint32_t kStageStep = C::kTileBytes >> 4;
    const uint32_t tq = tmem + C::kColQ;
    const uint32_t tdo = tmem + C::kColDO;
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) mma_commit(bar);
      __syncwarp();
    };
    int items = 0, tb = 0;  // items and blocks so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = sched_item(sched, k, G, cta, n_pairs, npairs, nb_max);
      if (item == -1) break;
      DqItem it;
      if (item < 0 || !dq_item_geom<D, PACKED>(p, item, nb_max, it)) continue;
      const int n = it.n;
      // Q_i and dO_i of this item in tensor memory (qdo_tmem: one completion per item; the
      // next needs qdo_free of this item, committed below after this wait).
      if (!(ok = warp_wait(qdo_tmem, items & 1, limit, abort_flag, kWaitDqQ))) break;
      if (!(ok = warp_wait(&k_full[tb % NS], (tb / NS) & 1, limit, abort_flag, kWaitDqK)))
        break;
      // S overwrites the previous item's last S, which the elementwise warps have read.
      if (tb > 0 && !(ok = warp_wait(s_free, (tb - 1) & 1, limit, abort_flag, kWaitDqSC)))
        break;
      tc_fence_after();
      if (elect_one()) {
        issue_rowdot_ts_d<D>(tmem + C::kColS, tq, dk + (tb % NS) * kStageStep, idesc_sq);
        mma_commit(s_full);
      }
      __syncwarp();
      // dP overwrites the previous item's last dP / dS: read by the elementwise warps and
      // by the last dQ product, which the tensor core runs before this one.
      if (!(ok = warp_wait(&v_full[tb % NS], (tb / NS) & 1, limit, abort_flag, kWaitDqV)))
        break;
      tc_fence_after();
      if (elect_one()) {
        issue_rowdot_ts_d<D>(tmem + C::kColDP, tdo, dv + (tb % NS) * kStageStep, idesc_sq);
        mma_commit(dp_full);
      }
      __syncwarp();
      if (n == 1) commit(qdo_free);  // every S and dP of the item issued
      for (int j = 0; ok && j < n; ++j) {
        const int b = tb + j, bn = b + 1;
        const int s = b % NS, sn = bn % NS;
        if (j + 1 < n) {
          if (!(ok = warp_wait(&k_full[sn], (bn / NS) & 1, limit, abort_flag, kWaitDqK) &&
                     warp_wait(s_free, b & 1, limit, abort_flag, kWaitDqSC)))
            break;
          tc_fence_after();
          if (elect_one()) {
            issue_rowdot_ts_d<D>(tmem + C::kColS, tq, dk + sn * kStageStep, idesc_sq);
            mma_commit(s_full);
          }
          __syncwarp();
        }
        if (!(ok = warp_wait(ds_full, b & 1, limit, abort_flag, kWaitDqDS))) break;
        // The first dQ product of an item overwrites the accumulator: the previous item's
        // epilogue must have read it (acc_free: one completion per item, each after an
        // acc_done that follows this wait).
        if (j == 0 && items > 0 &&
            !(ok = warp_wait(acc_free, (items - 1) & 1, limit, abort_flag, kWaitDqAccFree)))
          break;
        tc_fence_after();
        if (elect_one())
          issue_tmem_a_split_d(tmem + C::kColAcc0, tmem + C::kColDP, dk_mn + s * kStageStep,
                               idesc_acc, j > 0);
        __syncwarp();
        if (j + 1 < n) {
          if (!(ok = warp_wait(&v_full[sn], (bn / NS) & 1, limit, abort_flag, kWaitDqV)))
            break;
          tc_fence_after();
          if (elect_one()) {
            issue_rowdot_ts_d<D>(tmem + C::kColDP, tdo, dv + sn * kStageStep, idesc_sq);
            mma_commit(dp_full);
          }
          __syncwarp();
          if (j + 2 == n) commit(qdo_free);
        }
        commit(&kv_empty[s]);
      }
      if (!ok) break;
      commit(acc_done);
      tb += n;
      ++items;
    }
    commit(drain);
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitDqDrain);
  }
  else {
    // warps 0-7: thread = query row (TMEM lane); group g covers keys [64g, 64g + 64)
    const int g = warp >> 2;
    const int wq = warp & 3;
    const int c0 = g * 64;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::kColS + c0;
    const uint32_t t_dp = tmem + lane_base + C::kColDP + c0;
    const uint32_t t_row = tmem + lane_base + (g == 0 ? C::kColQ : C::kColDO);
    const uint32_t t_acc = tmem + lane_base + C::kColAcc0 + g * (D / 2);
    const float2 sl2x2 = make_float2(p.scale_log2, p.scale_log2);
    const uint8_t* gsrc = reinterpret_cast<const uint8_t*>(g == 0 ? p.in_q : p.in_do);
    int k = 0;
    // The next item of this CTA (false past the end).
    auto next_item = [&](DqItem& it) -> bool {
      for (;; ++k) {
        const int item = sched_item(sched, k, G, cta, n_pairs, npairs, nb_max);
        if (item == -1) return false;
        if (item >= 0 && dq_item_geom<D, PACKED>(p, item, nb_max, it)) {
          ++k;
          return true;
        }
      }
    };
    // This thread's row of Q_i (group 0) or dO_i (group 1) and its -L log2(e) and D
    // (rows past N: zeros, P = 0).
    auto fetch = [&](const DqItem& it, uint32_t (&rr)[D / 2], float& nl, float& dl) {
      const int row = it.i0 + wq * 32 + lane;
      nl = -INFINITY;
      dl = 0.f;
      if (row < it.N) {
        nl = -p.lse[it.sl.stat0 + row] * kLog2e;
        dl = p.delta[it.sl.stat0 + row];
      }
      load_row<D>(row < it.N ? gsrc + (it.sl.q_elem0 + (size_t)row * it.sl.row_elems) * 2
                             : nullptr,
                  rr, p.dh / 8);
    };
    // d = 64: this thread's staging row (16-byte chunks rotated by the lane, so that the
    // eight lanes of a quarter warp read eight different banks), then its L and D.
    auto stage_row = [&]() -> uint32_t {
      return smem_u32(smem) + C::kOffStage + (uint32_t)(warp * 32 + lane) * (D * 2);
    };
    auto stage_stat = [&]() -> uint32_t {
      return smem_u32(smem) + C::kOffStage + 256 * (D * 2) + (uint32_t)(warp * 32 + lane) * 8;
    };
    auto stage_issue = [&](const DqItem& it) {
      const int row = it.i0 + wq * 32 + lane;
      const bool in = row < it.N;
      const uint8_t* src =
          in ? gsrc + (it.sl.q_elem0 + (size_t)row * it.sl.row_elems) * 2 : gsrc;
      const int n16 = in ? p.dh / 8 : 0;
      const uint32_t dst = stage_row();
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        cp_async16(dst + ((c ^ (lane & 7)) & (D / 8 - 1)) * 16, src + (c < n16 ? c * 16 : 0),
                   c < n16 ? 16 : 0);
      const size_t si = in ? it.sl.stat0 + row : 0;
      cp_async4(stage_stat(), p.lse + si, in ? 4 : 0);
      cp_async4(stage_stat() + 4, p.delta + si, in ? 4 : 0);
      cp_async_commit();
    };
    auto stage_take = [&](const DqItem& it, uint32_t (&rr)[D / 2], float& nl, float& dl) {
      cp_async_wait_all();
      const uint32_t src = stage_row();
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = ld_shared_v4(src + ((c ^ (lane & 7)) & (D / 8 - 1)) * 16);
        rr[4 * c] = v.x;
        rr[4 * c + 1] = v.y;
        rr[4 * c + 2] = v.z;
        rr[4 * c + 3] = v.w;
      }
      const bool in = it.i0 + wq * 32 + lane < it.N;
      nl = in ? -__uint_as_float(ld_shared_u32(stage_stat())) * kLog2e : -INFINITY;
      dl = in ? __uint_as_float(ld_shared_u32(stage_stat() + 4)) : 0.f;
    };
    DqItem cur;
    bool have = next_item(cur);
    float neg_l2 = -INFINITY, dlt = 0.f;
    if (have) {
      uint32_t rr[D / 2];
      fetch(cur, rr, neg_l2, dlt);
      store_row_tmem<D>(rr, t_row);
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(qdo_tmem);
    }
    bool ok = true;
    int items = 0, tb = 0;  // items and blocks so far
    while (have) {
      const int row = cur.i0 + wq * 32 + lane;
      const float2 nl2x2 = make_float2(neg_l2, neg_l2);
      const float2 ndl2 = make_float2(-dlt, -dlt);
      DqItem nxt;
      bool have_next = false;
      float nl_next = -INFINITY, dl_next = 0.f;
      for (int j = 0; j < cur.n; ++j) {
        const int b = tb + j;
        if constexpr (C::kStageRows) {
          if (j == cur.n - 1) {  // the next item's rows, behind this last block's work
            // (the item is found again after the block: fewer registers live across it)
            const int k_here = k;
            DqItem ahead;
            if (next_item(ahead)) stage_issue(ahead);
            k = k_here;
          }
        }
        // ---- P = exp2(S * scale * log2(e) - L * log2(e)) for keys [c0, c0 + 64)
        if (!(ok = warp_wait(s_full, b & 1, limit, abort_flag, kWaitDqS))) break;
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64(t_s, sr);
        tc_fence_before();
        warp_arrive(s_free);
        float* pr = reinterpret_cast<float*>(sr);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 x = fma2(make_float2(pr[c], pr[c + 1]), sl2x2, nl2x2);
          pr[c] = ex2(x.x);
          pr[c + 1] = ex2(x.y);
        }
        const int kbase = j * kTileN + c0;  // key index of column 0 of this group
        if ((p.causal && kbase + 63 > cur.i0 + cur.off) || kbase + 64 > cur.Nk) {
          int lim = cur.Nk - 1 - kbase;                         // last key in range
          if (p.causal) lim = min(lim, row + cur.off - kbase);  // last key this row sees
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c > lim) pr[c] = 0.f;
        }
        // ---- dS = P * (dP - D), 16-bit pairs over dP
        if (!(ok = warp_wait(dp_full, b & 1, limit, abort_flag, kWaitDqDP))) break;
        tc_fence_after();
        uint32_t r[64];
        tmem_ld64(t_dp, r);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const float2 d = mul2(make_float2(pr[2 * u], pr[2 * u + 1]),
                                add2(make_float2(__uint_as_float(r[2 * u]),
                                                 __uint_as_float(r[2 * u + 1])),
                                     ndl2));
          r[u] = pack2<BF16>(d.x, d.y);  // in place: r[u] was read in this step or earlier
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
      tb += cur.n;
      // The next item's rows: loaded now, placed in tensor memory as soon as this item's
      // S and dP products have read the current ones (qdo_free: one completion per item,
      // committed after the item's last dP; the next needs the qdo_tmem arrival below).
      have_next = next_item(nxt);
      if (have_next) {
        uint32_t rr[D / 2];
        if constexpr (C::kStageRows)
          stage_take(nxt, rr, nl_next, dl_next);
        else
          fetch(nxt, rr, nl_next, dl_next);
        if (!(ok = warp_wait(qdo_free, items & 1, limit, abort_flag, kWaitDqQFree))) break;
        tc_fence_after();
        store_row_tmem<D>(rr, t_row);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(qdo_tmem);
      }
      // Epilogue: the accumulator into registers, released (acc_free), then dQ (scaled) to
      // HBM. Group g writes columns [g*d/2, (g+1)*d/2).
      if (!(ok = warp_wait(acc_done, items & 1, limit, abort_flag, kWaitDqDone))) break;
      tc_fence_after();
      uint32_t a[D / 2];
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc)
        tmem_ld32(t_acc + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&a[cc * 32]));
      tc_fence_before();
      warp_arrive(acc_free);
      if constexpr (kTmaOut) {
        // The warp's 32 rows x 32 columns staged in its 2 KiB buffer (64-byte rows, no
        // swizzle) and stored by one TMA copy once the buffer's previous store has read it.
        // A group whose columns all lie past the head dimension has nothing to store.
        if (g * (D / 2) < p.dh) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          uint8_t* buf = smem + C::kOffOut + warp * 2048;
          const uint32_t rbase = smem_u32(buf) + lane * 64;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              w4[i] = pack2<BF16>(__uint_as_float(a[8 * v + 2 * i]) * p.scale,
                                  __uint_as_float(a[8 * v + 2 * i + 1]) * p.scale);
            st_shared_v4(rbase + v * 16, w4[0], w4[1], w4[2], w4[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&map_dq, buf, g * (D / 2), cur.i0 + wq * 32, cur.sl.tma_bh);
            bulk_commit_group();
          }
        }
      } else if (row < cur.N) {
        uint8_t* drow = reinterpret_cast<uint8_t*>(p.out0) +
                        (cur.sl.q_elem0 + (size_t)row * cur.sl.row_elems) * 2 + g * D;
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc)
          store_row32<BF16>(drow + cc * 64, *reinterpret_cast<const uint32_t(*)[32]>(&a[cc * 32]),
                            p.scale, valid16(p.dh, g * (D / 2) + cc * 32, 4));
      }
      ++items;
      cur = nxt;
      have = have_next;
      neg_l2 = nl_next;
      dlt = dl_next;
    }
    if constexpr (C::kStageRows) cp_async_wait_all();  // no copy in flight at exit
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
