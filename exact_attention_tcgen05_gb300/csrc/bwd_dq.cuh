// bwd_dq.cuh - backward, dQ kernel: the grid runs over blocks of 128 query rows; each
// CTA owns dQ_i, streams every visible block of keys/values and accumulates
//   S = scale Q_i K_j^T, P = exp(S - L_i), dP = dO_i V_j^T, dS = P * (dP - D_i),
//   dQ_i += scale * dS K_j
// with no atomics ("Triton 05: Flash Attention", section 3단계 커널 구조, [3단계] dQ
// 커널: Q_i held on chip, loop over K_j, V_j; sections LSE로 P 재계산 and Softmax
// Gradient for the recomputation and the gradient). D_i comes from the preprocess
// kernel. The factor scale on dQ follows from S = scale Q K^T.
//
// Q_i and dO_i stay on chip as the A operands of S = Q_i K_j^T and dP = dO_i V_j^T, in
// tensor memory (each thread copies its own row there once, from global memory), so all
// three products read only their B operand (K_j or V_j) from shared memory, and shared
// memory holds just a three-block K/V ring.
// GB300 design: warps 0-3 and 4-7 are two softmax warpgroups that share each query row
// (thread = row = TMEM lane), group g taking keys [64g, 64g + 64) of a block; they turn
// S and dP (fp32 in tensor memory) into dS. Warp 8 is the TMA producer (Q_i and dO_i
// once, then a ring of K_j / V_j blocks), warp 9 issues the tcgen05 MMAs. Tensor memory:
// S (128 cols), dP (128 cols), dQ accumulator (d cols), Q_i and dO_i (d/2 cols each).
// Group g writes its dS pairs over
// dP columns [64g, 64g + 32), which feed dS K_j from tensor memory; S of the next block
// is computed while the softmax warps work on dP of this one.
#pragma once

#include "common.cuh"

namespace attn {

struct BwdParams {
  const void* in_q;    // [BH, N, d] Q (read directly by the dQ kernel)
  const void* in_k;    // [BH, N_k, d] K and V (read directly by the dK/dV kernel at d = 64)
  const void* in_v;
  const void* in_do;   // [BH, N, d] dO (read directly by the dQ kernel)
  const float* lse;    // [BH, N] natural-log L
  const float* delta;  // [BH, N] D
  void* out0;          // dQ (dQ kernel) or dK (dKV kernel)
  void* out1;          // dV (dKV kernel)
  int dh;              // head dimension of the tensors (<= D; columns past it read as zero)
  int N;               // query rows per slice (N_q; packed batches: per sequence, from vl)
  int Nk;              // key rows per slice (N_k); causal key j is visible to query i
                       // iff j <= i + (N_k - N_q)
  int causal;
  float scale;
  float scale_log2;    // scale * log2(e)
  unsigned long long wait_limit;
  int stall;           // failure tests: the TMA producer withholds every copy
  Varlen vl;           // packed variable-length batch (vl.cu_q == nullptr: dense)
};

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / kBoxCols;
  static constexpr int kTileBytes = kChunks * kBoxBytes;
  static constexpr int kStages = 2;
  static constexpr int kThreads = 320;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 256 + D;
  // Each CTA takes all 512 tensor-memory columns, so at most one may be resident per SM:
  // shared memory is padded past half of the SM's 228 KiB to guarantee that.
  static constexpr int kMinSmem = 120 * 1024;
};

template <int D>
struct DqCfg : BwdCfg<D> {
  using B = BwdCfg<D>;
  // Q_i and dO_i go straight from global memory to tensor memory, so shared memory holds
  // only the K/V ring: block j + S can be fetched as soon as dQ of block j (the last reader
  // of its K) has been issued and has finished. S = 3 at d = 128 (192 KiB), 4 at d = 64
  // (B2 H32 N8192 d64 on GB300: 1.371 -> 1.358 ms against 3).
  static constexpr int kStages = D == 64 ? 4 : 3;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * B::kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * B::kTileBytes;
  // k_full[S], v_full[S], kv_empty[S], s_full, s_free, dp_full, ds_full, acc_done, drain,
  // qdo_tmem
  static constexpr int kNumBars = 3 * kStages + 7;
  // Q_i and dO_i as 16-bit pairs in tensor memory (the A operands of S and dP):
  // d/2 columns each, after S, dP and the dQ accumulator (512 columns in all at d=128).
  static constexpr uint32_t kColQ = 256 + D, kColDO = 256 + D + D / 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes =
      (kOffMisc + 16 + 1024) > B::kMinSmem ? (kOffMisc + 16 + 1024) : B::kMinSmem;
};

// Writes 32 fp32 accumulator values, multiplied by `mul`, as 16-bit to a global row: the
// first n16 16-byte pieces (all four when the row is that wide).
template <bool BF16>
__device__ __forceinline__ void store_row32(uint8_t* dst, const uint32_t (&r)[32], float mul,
                                            int n16 = 4) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    pk[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < 4; ++v)
    if (v < n16) d4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
}

// K-major x K-major product over the head dimension: D[128 x 128] = A[128 x d] B[128 x d]^T.
template <int D>
__device__ __forceinline__ void issue_rowdot(uint32_t d_tmem, uint32_t a0, uint32_t b0,
                                             uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
    mma_ss(d_tmem, make_sdesc_sw128(a0 + off, 16, 1024), make_sdesc_sw128(b0 + off, 16, 1024),
           idesc, kk > 0 ? 1u : 0u);
  }
}


// Tensor-memory A [128 x 128] (16-bit pairs) times an MN-major [128 x d] tile in shared
// memory: D[128 x d] (+)= A B.
__device__ __forceinline__ void issue_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t b0,
                                             uint32_t idesc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 128 / 16; ++kk)
    mma_ts(d_tmem, a_tmem + kk * 8, make_sdesc_sw128(b0 + kk * 2048, kBoxBytes, 1024), idesc,
           (acc || kk > 0) ? 1u : 0u);
}

template <int D, bool BF16, bool PACKED>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q,
                       const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v,
                       const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
  using C = DqCfg<D>;
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
  uint64_t* qdo_tmem = drain + 1;  // Q_i and dO_i copied into tensor memory
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int bh = blockIdx.y;
  SliceRows sl;
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, sl)) return;
  const int N = sl.nq, Nk = sl.nk, off = sl.off;
  const int nb = (N + kTileM - 1) / kTileM;
  const int nkb = (Nk + kTileN - 1) / kTileN;
  if (PACKED && (int)blockIdx.x >= nb) return;  // past this sequence's query blocks
  const int ib = p.causal ? (nb - 1 - blockIdx.x) : blockIdx.x;  // longest first
  const int i0 = ib * kTileM;
  // key blocks 0 .. n-1 (causal: up to the block of the last key the tile's last row sees)
  const int n = p.causal ? min(nkb, (i0 + kTileM - 1 + off) / kTileN + 1) : nkb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 8);  // one arrival per softmax warp
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 8);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    mbar_init(qdo_tmem, 8);
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
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
    }
    int issued = 0;
    for (int j = 0; j < n; ++j) {
      const int s = j % NS;
      if (j >= NS &&
          !warp_wait(&kv_empty[s], ((j / NS) - 1) & 1, limit, abort_flag, kWaitDqEmpty))
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
      for (int j = max(0, issued - NS); j < issued; ++j) {
        mbar_wait(&k_full[j % NS], (j / NS) & 1, kDrainLimit, nullptr, kWaitDqDrain);
        mbar_wait(&v_full[j % NS], (j / NS) & 1, kDrainLimit, nullptr, kWaitDqDrain);
      }
    }
  } else if (warp == 9) {
    // MMA issuer: the warp runs the loop converged and waits in every lane; one elected
    // lane issues the MMAs and commits (a loop run by one lane alone loses issue slots to
    // the arithmetic warps of its SM sub-partition and starves the tensor core).
    const uint32_t idesc_sq = make_idesc(BF16, 128, kTileN, false, false);
    const uint32_t idesc_acc = make_idesc(BF16, 128, D, false, true);
    // Stage-0 descriptors: K (K-major, for S = Q K^T), K (MN-major, for dQ = dS K), V.
    const uint64_t dk = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dk_mn = make_sdesc_sw128(smem_u32(smem + C::kOffK), kBoxBytes, 1024);
    const uint64_t dv = make_sdesc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
    constexpr uint32_t kStageStep = C::kTileBytes >> 4;
    const uint32_t tq = tmem + C::kColQ;
    const uint32_t tdo = tmem + C::kColDO;
    bool ok = warp_wait(qdo_tmem, 0, limit, abort_flag, kWaitDqQ) &&
              warp_wait(&k_full[0], 0, limit, abort_flag, kWaitDqK);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        issue_rowdot_ts_d<D>(tmem + C::kColS, tq, dk, idesc_sq);
        mma_commit(s_full);
      }
      __syncwarp();
      ok = warp_wait(&v_full[0], 0, limit, abort_flag, kWaitDqV);
    }
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        issue_rowdot_ts_d<D>(tmem + C::kColDP, tdo, dv, idesc_sq);
        mma_commit(dp_full);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n; ++j) {
      const int s = j % NS;
      const int jn = j + 1;
      const int sn = jn % NS;
      if (jn < n) {
        // S of the next block overwrites S once the softmax warps have read it.
        if (!(ok = warp_wait(&k_full[sn], (jn / NS) & 1, limit, abort_flag, kWaitDqK) &&
                   warp_wait(s_free, j & 1, limit, abort_flag, kWaitDqSC)))
          break;
        tc_fence_after();
        if (elect_one()) {
          issue_rowdot_ts_d<D>(tmem + C::kColS, tq, dk + sn * kStageStep, idesc_sq);
          mma_commit(s_full);
        }
        __syncwarp();
      }
      if (!(ok = warp_wait(ds_full, j & 1, limit, abort_flag, kWaitDqDS))) break;
      tc_fence_after();
      // dQ_i += dS K_j (dS read from tensor memory, over dP)
      if (elect_one())
        issue_tmem_a_split_d(tmem + C::kColAcc0, tmem + C::kColDP, dk_mn + s * kStageStep,
                             idesc_acc, j > 0);
      __syncwarp();
      if (jn < n) {
        if (!(ok = warp_wait(&v_full[sn], (jn / NS) & 1, limit, abort_flag, kWaitDqV))) break;
        tc_fence_after();
        if (elect_one()) {
          issue_rowdot_ts_d<D>(tmem + C::kColDP, tdo, dv + sn * kStageStep, idesc_sq);
          mma_commit(dp_full);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(&kv_empty[s]);
      __syncwarp();
    }
    if (elect_one()) {
      if (ok) mma_commit(acc_done);
      mma_commit(drain);
    }
    __syncwarp();
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitDqDrain);
  } else {
    // warps 0-7: thread = query row (TMEM lane); group g covers keys [64g, 64g + 64)
    const int g = warp >> 2;
    const int wq = warp & 3;
    const int c0 = g * 64;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::kColS + c0;
    const uint32_t t_dp = tmem + lane_base + C::kColDP + c0;
    const int row = i0 + wq * 32 + lane;
    const float2 sl2x2 = make_float2(p.scale_log2, p.scale_log2);
    float neg_l2 = -INFINITY;  // -L * log2(e); rows past N get P = 0
    float dlt = 0.f;
    if (row < N) {
      neg_l2 = -p.lse[sl.stat0 + row] * kLog2e;
      dlt = p.delta[sl.stat0 + row];
    }
    const float2 nl2x2 = make_float2(neg_l2, neg_l2);
    const float2 ndl2 = make_float2(-dlt, -dlt);
    // Group 0 copies this row of Q_i, group 1 the row of dO_i, into tensor memory
    // (rows past N as zeros).
    bool ok = true;
    {
      const uint8_t* gsrc = reinterpret_cast<const uint8_t*>(g == 0 ? p.in_q : p.in_do);
      copy_row_to_tmem<D>(row < N ? gsrc + (sl.q_elem0 + (size_t)row * sl.row_elems) * 2
                                  : nullptr,
                          tmem + lane_base + (g == 0 ? C::kColQ : C::kColDO), p.dh / 8);
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(qdo_tmem);
    }
    for (int j = 0; ok && j < n; ++j) {
      // ---- P = exp2(S * scale * log2(e) - L * log2(e)) for keys [c0, c0 + 64)
      if (!(ok = warp_wait(s_full, j & 1, limit, abort_flag, kWaitDqS))) break;
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
      if ((p.causal && kbase + 63 > i0 + off) || kbase + 64 > Nk) {  // diagonal or ragged
        int lim = Nk - 1 - kbase;                       // last key in range
        if (p.causal) lim = min(lim, row + off - kbase);  // last key this row sees
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c > lim) pr[c] = 0.f;
      }
      // ---- dS = P * (dP - D), 16-bit pairs over dP
      if (!(ok = warp_wait(dp_full, j & 1, limit, abort_flag, kWaitDqDP))) break;
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
    if (ok && warp_wait(acc_done, 0, limit, abort_flag, kWaitDqDone)) {
      tc_fence_after();
      // Group g writes columns [g*d/2, (g+1)*d/2) of dQ, scaled.
      uint8_t* drow = reinterpret_cast<uint8_t*>(p.out0) +
                      (sl.q_elem0 + (size_t)row * sl.row_elems) * 2 + g * D;
      const uint32_t t_acc = tmem + lane_base + C::kColAcc0 + g * (D / 2);
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t a[32];
        tmem_ld32(t_acc + cc * 32, a);
        if (row < N)
          store_row32<BF16>(drow + cc * 64, a, p.scale, valid16(p.dh, g * (D / 2) + cc * 32, 4));
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
