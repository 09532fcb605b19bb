// bwd_dkv.cuh - backward, dK/dV kernel: the grid runs over blocks of 128 keys; each CTA
// owns dK_j and dV_j, keeps K_j and V_j on chip and streams every query block that sees
// them ("Triton 05: Flash Attention", section 3단계 커널 구조, [2단계] dKV 커널: K_j, V_j
// fixed in SRAM, loop over all Q_i; no atomics because each CTA owns its outputs).
//
// It works in the transposed orientation so that the key index runs down the tensor
// memory lanes: per query block i
//   S^T = scale K_j Q_i^T,  P^T = exp(S^T - L_i),  dV_j += P^T dO_i,
//   dP^T = V_j dO_i^T,      dS^T = P^T * (dP^T - D_i),  dK_j += scale * dS^T Q_i.
// P^T and dS^T are written back over S^T and dP^T as 16-bit pairs and used as the A
// operand of the two accumulating products straight from tensor memory.
//
// Roles (10 warps): warps 0-3 and 4-7 are two softmax warpgroups that share each key row
// (thread = key row = TMEM lane); group g handles queries [64g, 64g + 64) of the block, so
// a thread does 64 exponentials per block and every SM sub-partition runs two softmax
// warps. Group g writes its 16-bit pairs into columns [64g, 64g + 32) of the region it
// read, where no other thread reads. Warp 8: TMA producer; warp 9: MMA issuer.
// Tensor memory: S^T (128 cols), dP^T (128), dV (d), dK (d).
#pragma once

#include "bwd_dq.cuh"

namespace attn {

template <int D>
struct DkvCfg : BwdCfg<D> {
  using B = BwdCfg<D>;
  static constexpr int kThreads = 320;
  // Q/dO ring depth: three blocks at d = 64 (measured on GB300 against two: GPT-2-medium
  // shape 0.441 -> 0.428 ms, B2 H32 N8192 d64 2.081 -> 1.986; four ran 1-1.5% slower than
  // three), two at d = 128, where shared memory has no room for more.
  static constexpr int kStages = D == 64 ? 3 : 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + B::kTileBytes;
  static constexpr int kOffQ = kOffV + B::kTileBytes;
  static constexpr int kOffDO = kOffQ + kStages * B::kTileBytes;
  static constexpr int kOffStats = kOffDO + kStages * B::kTileBytes;  // 2 x (128 + 128) f32
  static constexpr int kOffBar = kOffStats + 2 * 256 * 4;
  // kv_full, q_full[S], do_full[S], qdo_empty[S], s_full, p_full, dp_full, ds_full,
  // acc_done, drain, stats_ready[2]
  static constexpr int kNumBars = 1 + 3 * kStages + 8;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes =
      (kOffMisc + 16 + 1024) > B::kMinSmem ? (kOffMisc + 16 + 1024) : B::kMinSmem;
  // d = 64 (KV_TMEM): K_j and V_j also fit in tensor memory (d/2 columns of 16-bit pairs
  // each, after S^T, dP^T, dV and dK: 448 of 512), so S^T = K_j Q_i^T and dP^T = V_j dO_i^T
  // run as TS products (A from tensor memory), which read only B from shared memory
  // (measured on GB300: B2 H32 N8192 d64 dK/dV 2.236 -> 2.049 ms). Each elementwise thread
  // copies its own key row there once, which costs start-up latency; the launcher picks
  // this form only when a key block meets enough query blocks. At d = 128 the four
  // accumulators fill all 512 columns.
  static constexpr uint32_t kColK = 256 + 2 * D, kColV = 256 + 2 * D + D / 2;
};

template <int D, bool BF16, bool PACKED, bool KV_TMEM>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
  using C = DkvCfg<D>;
  static_assert(!KV_TMEM || D == 64, "K and V fit in tensor memory only at d = 64");
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* do_full = q_full + NS;
  uint64_t* qdo_empty = do_full + NS;
  uint64_t* s_full = qdo_empty + NS;
  uint64_t* p_full = s_full + 1;
  uint64_t* dp_full = p_full + 1;
  uint64_t* ds_full = dp_full + 1;
  uint64_t* acc_done = ds_full + 1;
  uint64_t* drain = acc_done + 1;
  uint64_t* stats_ready = drain + 1;  // [2], one per statistics buffer
  float* stats = reinterpret_cast<float*>(smem + C::kOffStats);  // [2][-L*log2e x128, D x128]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int bh = blockIdx.y;
  SliceRows sl;
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, sl)) return;
  const int N = sl.nq, Nk = sl.nk, off = sl.off;
  const int jb = blockIdx.x;  // causal: block 0 sees the most query blocks, so runs first
  if (PACKED && jb * kTileN >= Nk) return;  // past this sequence's keys
  const int j0 = jb * kTileN;
  if (PACKED && N == 0) {
    // A packed sequence with keys but no queries: no query sees these keys, so their
    // gradients are zero.
    const int rows = min(kTileN, Nk - j0);
    const int kVec = p.dh / 8;  // 16-byte pieces per row
    for (int idx = threadIdx.x; idx < 2 * rows * kVec; idx += blockDim.x) {
      const int t = idx / (rows * kVec), r = (idx / kVec) % rows, c = idx % kVec;
      uint8_t* base = reinterpret_cast<uint8_t*>(t == 0 ? p.out0 : p.out1);
      reinterpret_cast<uint4*>(base + (sl.k_elem0 + (size_t)(j0 + r) * sl.row_elems) * 2)[c] =
          make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int nb = (N + kTileM - 1) / kTileM;
  // causal: the first query block with a row that sees key j0 (row + off >= j0)
  const int i_first = (p.causal && j0 > off) ? (j0 - off) / kTileM : 0;
  const int n = nb - i_first;  // query blocks i_first .. nb-1

  if (threadIdx.x == 0) {
    mbar_init(kv_full, KV_TMEM ? 8 : 1);  // elementwise warps (8) or TMA (1)
    for (int s = 0; s < NS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&do_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 8);  // one arrival per softmax warp
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 8);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    mbar_init(&stats_ready[0], 8);
    mbar_init(&stats_ready[1], 8);
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
    // TMA producer. The warp runs converged (waits in every lane); the elected lane issues.
    if (elect_one()) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      tma_prefetch_map(&map_do);
      if constexpr (!KV_TMEM) {
        mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_rows<PACKED>(smem + C::kOffK + c * kBoxBytes, &map_k, kv_full,
                                c * kBoxCols, j0, sl, true);
          tma_load_rows<PACKED>(smem + C::kOffV + c * kBoxBytes, &map_v, kv_full,
                                c * kBoxCols, j0, sl, true);
        }
      }
    }
    __syncwarp();
    int issued = 0;
    for (int it = 0; it < n; ++it) {
      const int s = it % NS;
      const int i = i_first + it;
      if (it >= NS &&
          !warp_wait(&qdo_empty[s], ((it / NS) - 1) & 1, limit, abort_flag, kWaitDkvEmpty))
        break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&q_full[s], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffQ + s * C::kTileBytes + c * kBoxBytes, &map_q,
                                &q_full[s], c * kBoxCols, i * kTileM, sl, false);
        mbar_arrive_expect_tx(&do_full[s], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffDO + s * C::kTileBytes + c * kBoxBytes, &map_do,
                                &do_full[s], c * kBoxCols, i * kTileM, sl, false);
      }
      __syncwarp();
      issued = it + 1;
    }
    if (*abort_flag) {
      if constexpr (!KV_TMEM) mbar_wait(kv_full, 0, kDrainLimit, nullptr, kWaitDkvDrain);
      for (int it = max(0, issued - NS); it < issued; ++it) {
        mbar_wait(&q_full[it % NS], (it / NS) & 1, kDrainLimit, nullptr, kWaitDkvDrain);
        mbar_wait(&do_full[it % NS], (it / NS) & 1, kDrainLimit, nullptr, kWaitDkvDrain);
      }
    }
  } else if (warp == 9) {
    // MMA issuer: converged warp, elected lane issues (see the dQ kernel).
    const uint32_t idesc_st = make_idesc(BF16, 128, kTileM, false, false);
    const uint32_t idesc_acc = make_idesc(BF16, 128, D, false, true);
    const uint64_t dk = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dv = make_sdesc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
    const uint64_t dq = make_sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t ddo = make_sdesc_sw128(smem_u32(smem + C::kOffDO), 16, 1024);
    const uint64_t dq_mn = make_sdesc_sw128(smem_u32(smem + C::kOffQ), kBoxBytes, 1024);
    const uint64_t ddo_mn = make_sdesc_sw128(smem_u32(smem + C::kOffDO), kBoxBytes, 1024);
    constexpr uint32_t kStageStep = C::kTileBytes >> 4;
    // S^T = K_j Q_i^T and dP^T = V_j dO_i^T, with K_j / V_j from shared or tensor memory.
    auto issue_st = [&](int stage) {
      if constexpr (KV_TMEM)
        issue_rowdot_ts_d<D>(tmem + C::kColS, tmem + C::kColK, dq + stage * kStageStep,
                             idesc_st);
      else
        issue_rowdot_d<D>(tmem + C::kColS, dk, dq + stage * kStageStep, idesc_st);
    };
    auto issue_dpt = [&](int stage) {
      if constexpr (KV_TMEM)
        issue_rowdot_ts_d<D>(tmem + C::kColDP, tmem + C::kColV, ddo + stage * kStageStep,
                             idesc_st);
      else
        issue_rowdot_d<D>(tmem + C::kColDP, dv, ddo + stage * kStageStep, idesc_st);
    };
    bool ok = warp_wait(kv_full, 0, limit, abort_flag, kWaitDkvKV) &&
              warp_wait(&q_full[0], 0, limit, abort_flag, kWaitDkvQ);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        issue_st(0);
        mma_commit(s_full);
      }
      __syncwarp();
      ok = warp_wait(&do_full[0], 0, limit, abort_flag, kWaitDkvDO);
    }
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        issue_dpt(0);
        mma_commit(dp_full);
      }
      __syncwarp();
    }
    for (int it = 0; ok && it < n; ++it) {
      const int s = it % NS;
      const int in = it + 1;
      const int sn = in % NS;
      if (!(ok = warp_wait(p_full, it & 1, limit, abort_flag, kWaitDkvP))) break;
      tc_fence_after();
      // dV_j += P^T dO_i
      if (elect_one())
        issue_tmem_a_split_d(tmem + C::kColAcc0, tmem + C::kColS, ddo_mn + s * kStageStep,
                             idesc_acc, it > 0);
      __syncwarp();
      if (in < n) {
        if (!(ok = warp_wait(&q_full[sn], (in / NS) & 1, limit, abort_flag, kWaitDkvQ))) break;
        tc_fence_after();
        if (elect_one()) {
          issue_st(sn);
          mma_commit(s_full);
        }
        __syncwarp();
      }
      if (!(ok = warp_wait(ds_full, it & 1, limit, abort_flag, kWaitDkvDS))) break;
      tc_fence_after();
      // dK_j += dS^T Q_i
      if (elect_one())
        issue_tmem_a_split_d(tmem + C::kColAcc1, tmem + C::kColDP, dq_mn + s * kStageStep,
                             idesc_acc, it > 0);
      __syncwarp();
      if (in < n) {
        if (!(ok = warp_wait(&do_full[sn], (in / NS) & 1, limit, abort_flag, kWaitDkvDO)))
          break;
        tc_fence_after();
        if (elect_one()) {
          issue_dpt(sn);
          mma_commit(dp_full);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(&qdo_empty[s]);
      __syncwarp();
    }
    if (elect_one()) {
      if (ok) mma_commit(acc_done);
      mma_commit(drain);
    }
    __syncwarp();
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitDkvDrain);
  } else {
    // warps 0-7: thread = key row (TMEM lane); group g covers queries [64g, 64g + 64)
    const int g = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // 0..127
    const int key = j0 + row;
    const int c0 = g * 64;           // first query column of this group
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::kColS + c0;
    const uint32_t t_dp = tmem + lane_base + C::kColDP + c0;
    const float2 sl2x2 = make_float2(p.scale_log2, p.scale_log2);
    // Group 0 stages -L*log2(e), group 1 stages D: one value per thread per query block.
    const float* src = (g == 0 ? p.lse : p.delta) + sl.stat0;
    auto load_stat = [&](int i) -> float {
      const int q = i * kTileM + row;
      if (q >= N) return g == 0 ? -INFINITY : 0.f;  // padding queries: P = 0, D = 0
      const float x = src[q];
      return g == 0 ? -x * kLog2e : x;
    };
    float stat_next = load_stat(i_first);  // issued first: its latency overlaps the copy
    if constexpr (KV_TMEM) {
      // Group 0 copies this key's row of K_j, group 1 its row of V_j, into tensor memory
      // (keys past the slice's end as zeros); the MMA warp waits for all eight warps.
      const uint8_t* gsrc = reinterpret_cast<const uint8_t*>(g == 0 ? p.in_k : p.in_v);
      copy_row_to_tmem<D>(key < Nk ? gsrc + (sl.k_elem0 + (size_t)key * sl.row_elems) * 2
                                   : nullptr,
                          tmem + lane_base + (g == 0 ? C::kColK : C::kColV), p.dh / 8);
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(kv_full);
    }
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      const int i = i_first + it;
      // Double-buffered statistics: buffer it&1 was last read in iteration it-2, and
      // every thread has passed iteration it-1's stats_ready wait, which needs all eight
      // warps' arrivals, so nobody still reads it.
      float* st = stats + (it & 1) * 256;
      st[g * 128 + row] = stat_next;
      warp_arrive(&stats_ready[it & 1]);
      if (it + 1 < n) stat_next = load_stat(i + 1);
      if (!(ok = warp_wait(&stats_ready[it & 1], (it >> 1) & 1, limit, abort_flag,
                           kWaitDkvStats)))
        break;

      // ---- P^T = exp2(S^T * scale * log2(e) - L * log2(e)), 16-bit pairs over S^T
      if (!(ok = warp_wait(s_full, it & 1, limit, abort_flag, kWaitDkvS))) break;
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
        const float2 b = fma2(make_float2(pr[4 * c4 + 2], pr[4 * c4 + 3]), sl2x2,
                              make_float2(nl.z, nl.w));
        pr[4 * c4] = ex2(a.x);
        pr[4 * c4 + 1] = ex2(a.y);
        pr[4 * c4 + 2] = ex2(b.x);
        pr[4 * c4 + 3] = ex2(b.y);
      }
      if (p.causal && i * kTileM + off < j0 + kTileN - 1) {
        // A block on the diagonal: query i*128 + c0 + c sees this key iff
        // i*128 + c0 + c + off >= key, i.e. c >= key - off - i*128 - c0.
        const int first = key - off - i * kTileM - c0;
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
      if (!(ok = warp_wait(dp_full, it & 1, limit, abort_flag, kWaitDkvDP))) break;
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
        // Pack in place: r[2u] and r[2u+1] were read in this step (u = 0) or earlier.
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
    if (ok && warp_wait(acc_done, 0, limit, abort_flag, kWaitDkvDone)) {
      tc_fence_after();
      // Group 0 writes dV, group 1 writes dK (scaled).
      uint8_t* dst = reinterpret_cast<uint8_t*>(g == 0 ? p.out1 : p.out0) +
                     (sl.k_elem0 + (size_t)key * sl.row_elems) * 2;
      const uint32_t t_acc = tmem + lane_base + (g == 0 ? C::kColAcc0 : C::kColAcc1);
      const float mul = (g == 0) ? 1.f : p.scale;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t a[32];
        tmem_ld32(t_acc + cc * 32, a);
        if (key < Nk) store_row32<BF16>(dst + cc * 64, a, mul, valid16(p.dh, cc * 32, 4));
      }
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
