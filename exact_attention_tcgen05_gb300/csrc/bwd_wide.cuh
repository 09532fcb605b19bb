// bwd_wide.cuh - the backward for head dimensions above 128 (up to 256): the recomputing
// backward of bwd_dq.cuh and bwd_dkv.cuh ("Triton 05: Flash Attention", sections LSE로 P
// 재계산, Softmax Gradient and 3단계 커널 구조: P = exp(S - L), dV = P^T dO,
// dP = dO V^T, dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q, no atomics) on the
// tile shape of fwd_wide.cuh.
//
// At d = 256 the accumulators of dK and dV together take all 512 tensor-memory columns,
// and 128 x 256 tiles take 64 KiB of shared memory each, so the three outputs come from
// three passes of one kernel template, each a CTA per 128 rows of one (b, h) slice that
// keeps one or two 128 x 256 tiles resident and streams 64-row blocks of two others:
//   dQ: rows = queries; Q_i, dO_i resident; K_j, V_j streamed;
//       S = Q_i K_j^T, dP = dO_i V_j^T, dS = P * (dP - D_i), dQ_i += dS K_j;
//   dK: rows = keys; K_j, V_j resident; Q_i, dO_i streamed;
//       S^T = K_j Q_i^T, dP^T = V_j dO_i^T, dS^T = P^T * (dP^T - D_i), dK_j += dS^T Q_i;
//   dV: rows = keys; K_j resident; Q_i, dO_i streamed;
//       S^T = K_j Q_i^T, dV_j += P^T dO_i.
// dQ and dK carry the factor scale (applied when they are stored). S^T is computed in both
// key passes (five products per pair of blocks instead of four): the price of fitting.
// Numerics as in the 128-column kernels: P in fp32 from the natural-log L, dS from that P,
// each rounded once to the input type as the A operand of its product.
//
// Roles: warps 0-3 elementwise, one row per thread (TMEM lane); warp 4 TMA producer; warp
// 5 MMA issuer and tensor-memory owner. In dQ and dK the first resident tile (Q_i or K_j)
// sits in shared memory and the second (dO_i, V_j) is copied by the elementwise threads, a
// row each, into tensor memory, where it is the A operand of dP; in dV the only resident
// tile, K_j, is copied there likewise and is the A operand of S^T. An A operand in shared
// memory is re-read for every 16-column step, which for these 64-column products costs
// more shared-memory bandwidth than the B operand (measured on GB300: an S step with A in
// shared memory issues in ~56 cycles, one with A in tensor memory in ~42). Shared memory
// holds three stages of X (the B operand of S) and two of Y (of dP; of the accumulation
// in dV), each stage freed by its last product: X by the accumulation (dQ, dK) or by S
// (dV), Y by dP (dQ, dK) or by the accumulation (dV). Tensor memory: S (two buffers in
// dV, where P is written over S and nothing else needs columns), dP, the 256-column
// accumulator and the copied tile: S(b + 1) runs while the elementwise warps finish
// block b.
#pragma once

#include "bwd_dq.cuh"
#include "launch.h"

namespace attn {

enum WideMode : int { kWideDQ = 0, kWideDK = 1, kWideDV = 2 };

template <int MODE>
struct BwdWCfg {
  static constexpr int D = 256;
  static constexpr int kBN = 64;                       // streamed rows per block
  static constexpr int kChunks = D / kBoxCols;         // 4
  static constexpr int kTileBytes = kChunks * kBoxBytes;  // resident 128 x 256 tile: 64 KiB
  static constexpr int kBlkBox = kBN * 128;             // [64 x 64] box: 8 KiB
  static constexpr int kBlkBytes = kChunks * kBlkBox;   // streamed 64 x 256 block: 32 KiB
  static constexpr bool kDV = MODE == kWideDV;
  static constexpr bool kA2Tmem = !kDV;  // dQ, dK: the second resident tile in tensor memory
  static constexpr bool kA1Tmem = kDV;   // dV: the resident tile in tensor memory
  static constexpr int kSBufs = kDV ? 2 : 1;  // S buffers
  // Streamed X (the B operand of S) and Y (of dP, or of the accumulating product in dV)
  static constexpr int kXStages = 3;
  static constexpr int kYStages = 2;
  static constexpr int kOffA = 0;
  static constexpr int kOffX = kOffA + kTileBytes;
  static constexpr int kOffY = kOffX + kXStages * kBlkBytes;
  static constexpr int kOffStats = kOffY + kYStages * kBlkBytes;  // [2][-L log2 e x64, D x64]
  static constexpr int kOffBar = kOffStats + 2 * 128 * 4;
  // a_full, a2_tmem, x_full[XS], x_empty[XS], y_full[YS], y_empty[YS], s_full[2], s_free,
  // dp_full, ds_full[2] (dV: P written), stats_ready[2], acc_last, drain
  static constexpr int kNumBars = 2 + 2 * kXStages + 2 * kYStages + 2 + 1 + 1 + 2 + 2 + 1 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kSmemBytes > 114 * 1024, "two CTAs could share an SM");
  static constexpr int kThreads = 192;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;     // S buffer b at 64 b (P over its first 32 in dV)
  static constexpr uint32_t kColDP = 64;   // dQ, dK: dP (dS over its first 32 columns)
  static constexpr uint32_t kColAcc = 128;
  static constexpr uint32_t kColA2 = 384;  // the copied tile (dO_i, V_j, K_j) as 16-bit pairs
};

// Maps: a1 = the resident tile in shared memory (128-row boxes), x/y = streamed blocks
// (64-row boxes). dQ and dK read the second resident tile's rows from p.in_do / p.in_v.
// PACKED: slices are (sequence, head) pairs of a packed batch (common.cuh, SliceRows); a
// tile past its sequence's end does nothing, and a sequence with keys but no queries gets
// zero key gradients.
template <int MODE, bool BF16, bool PACKED>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_wide_kernel(const __grid_constant__ CUtensorMap map_a1,
                         const __grid_constant__ CUtensorMap map_x,
                         const __grid_constant__ CUtensorMap map_y, const BwdParams p) {
  using C = BwdWCfg<MODE>;
  constexpr bool kDV = C::kDV;
  constexpr bool kRowsAreQueries = MODE == kWideDQ;
  constexpr int NX = C::kXStages, NY = C::kYStages, NB = C::kSBufs;
  constexpr int kBN = C::kBN;
  // Wait-site codes: the dQ kernel's for the dQ pass, the dK/dV kernel's for the others.
  constexpr int kSiteA = kRowsAreQueries ? kWaitDqQ : kWaitDkvKV;
  constexpr int kSiteX = kRowsAreQueries ? kWaitDqK : kWaitDkvQ;
  constexpr int kSiteY = kRowsAreQueries ? kWaitDqV : kWaitDkvDO;
  constexpr int kSiteEmpty = kRowsAreQueries ? kWaitDqEmpty : kWaitDkvEmpty;
  constexpr int kSiteS = kRowsAreQueries ? kWaitDqS : kWaitDkvS;
  constexpr int kSiteDP = kRowsAreQueries ? kWaitDqDP : kWaitDkvDP;
  constexpr int kSiteDS = kRowsAreQueries ? kWaitDqDS : kWaitDkvDS;
  constexpr int kSiteDone = kRowsAreQueries ? kWaitDqDone : kWaitDkvDone;
  constexpr int kSiteDrain = kRowsAreQueries ? kWaitDqDrain : kWaitDkvDrain;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* a_full = bars;
  uint64_t* a2_tmem = bars + 1;  // dQ, dK: every elementwise warp has copied its rows
  uint64_t* x_full = bars + 2;
  uint64_t* x_empty = x_full + NX;
  uint64_t* y_full = x_empty + NX;
  uint64_t* y_empty = y_full + NY;
  uint64_t* s_full = y_empty + NY;    // [NB] per S buffer
  uint64_t* s_free = s_full + 2;      // dQ, dK: S has been read (one buffer)
  uint64_t* dp_full = s_free + 1;
  uint64_t* ds_full = dp_full + 1;    // [NB] dS (dV: P) of the buffer's block is written
  uint64_t* stats_ready = ds_full + 2;  // [2] per statistics buffer
  uint64_t* acc_last = stats_ready + 2;  // the last accumulating product
  uint64_t* drain = acc_last + 1;
  float* stats = reinterpret_cast<float*>(smem + C::kOffStats);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int bh = blockIdx.y;
  SliceRows sl;
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, sl)) return;
  const int N = sl.nq, Nk = sl.nk, off = sl.off;
  // Rows of this CTA and the streamed blocks it visits (b0 .. b0 + n - 1).
  const int n_rows = kRowsAreQueries ? N : Nk;
  const int n_tiles = (n_rows + kTileM - 1) / kTileM;
  if (PACKED && (int)blockIdx.x >= n_tiles) return;  // past this sequence's rows
  const int r0 = (n_tiles - 1 - (int)blockIdx.x) * kTileM;  // longest first within a head
  int b0, n;
  if constexpr (kRowsAreQueries) {
    // keys up to the block of the last key the tile's last query sees
    const int nkb = (Nk + kBN - 1) / kBN;
    b0 = 0;
    n = p.causal ? min(nkb, (r0 + kTileM - 1 + off) / kBN + 1) : nkb;
  } else {
    // queries from the block of the first query that sees the tile's first key
    const int nqb = (N + kBN - 1) / kBN;
    b0 = (p.causal && r0 > off) ? (r0 - off) / kBN : 0;
    n = nqb - b0;  // >= 1 unless the slice has no queries: the last query sees every key
  }

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a2_tmem, 4);  // one arrival per elementwise warp
    for (int s = 0; s < NX; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], 1);
    }
    for (int s = 0; s < NY; ++s) {
      mbar_init(&y_full[s], 1);
      mbar_init(&y_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&ds_full[b], 4);      // one arrival per elementwise warp
      mbar_init(&stats_ready[b], 4);  // one arrival per elementwise warp
    }
    mbar_init(s_free, 4);
    mbar_init(dp_full, 1);
    mbar_init(acc_last, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint64_t limit = p.wait_limit;
  // Row of the resident tiles and of the streamed blocks in the slice: queries or keys.
  const bool a_keys = !kRowsAreQueries, x_keys = kRowsAreQueries;

  if (warp == 4 && p.stall) {
    // Failure tests: the producer withholds every copy; the consumers' waits run out.
  } else if (warp == 4) {
    // ------------------------------ TMA producer ------------------------------
    if (n > 0 && elect_one()) {
      tma_prefetch_map(&map_x);
      tma_prefetch_map(&map_y);
      if (!C::kA1Tmem) {
        tma_prefetch_map(&map_a1);
        mbar_arrive_expect_tx(a_full, C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffA + c * kBoxBytes, &map_a1, a_full, c * kBoxCols,
                                r0, sl, a_keys);
      }
    }
    __syncwarp();
    // X(b) into stage b % NX once the stage's previous block is released (x_empty), Y(b)
    // likewise; each empty barrier completes once per block of its stage, after a copy
    // issued past its wait. Order: X(0), X(1), then Y(b), X(b + 2). It never waits on a
    // product that needs a later copy: Y(b) waits for a product of block b - 2, X(b + 2)
    // for one of block b - 1 (the accumulation in dQ/dK, S in dV), and neither of those
    // needs more than X(b) and Y(b - 1).
    int x_issued = 0, y_issued = 0;
    auto load_x = [&](int b) -> bool {
      const int s = b % NX;
      if (b >= NX &&
          !warp_wait(&x_empty[s], ((b / NX) - 1) & 1, limit, abort_flag, kSiteEmpty))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(&x_full[s], C::kBlkBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffX + s * C::kBlkBytes + c * C::kBlkBox, &map_x,
                               &x_full[s], c * kBoxCols, (b0 + b) * kBN, sl, x_keys);
      }
      __syncwarp();
      x_issued = b + 1;
      return true;
    };
    auto load_y = [&](int b) -> bool {
      const int s = b % NY;
      if (b >= NY &&
          !warp_wait(&y_empty[s], ((b / NY) - 1) & 1, limit, abort_flag, kSiteEmpty))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(&y_full[s], C::kBlkBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffY + s * C::kBlkBytes + c * C::kBlkBox, &map_y,
                               &y_full[s], c * kBoxCols, (b0 + b) * kBN, sl, x_keys);
      }
      __syncwarp();
      y_issued = b + 1;
      return true;
    };
    bool ok = true;
    constexpr int kLead = NX - 1;  // X copies ahead of Y
    for (int b = 0; ok && b < min(kLead, n); ++b) ok = load_x(b);
    for (int b = 0; ok && b < n; ++b) {
      ok = load_y(b);
      if (ok && b + kLead < n) ok = load_x(b + kLead);
    }
    if (*abort_flag) {
      // Let every copy this CTA started land before its shared memory is released.
      if (n > 0 && !C::kA1Tmem) mbar_wait(a_full, 0, kDrainLimit, nullptr, kSiteDrain);
      for (int b = max(0, x_issued - NX); b < x_issued; ++b)
        mbar_wait(&x_full[b % NX], (b / NX) & 1, kDrainLimit, nullptr, kSiteDrain);
      for (int b = max(0, y_issued - NY); b < y_issued; ++b)
        mbar_wait(&y_full[b % NY], (b / NY) & 1, kDrainLimit, nullptr, kSiteDrain);
    }
  } else if (warp == 5) {
    // ------------------------------ MMA issuer --------------------------------
    // dV, per block b: S(b + 1) into the other S buffer (its previous P was read by the
    // accumulation of b - 1, issued before: the tensor core runs them in order), then
    // dV += P(b) Y(b) once P is written. dQ/dK, per block b: S(b + 1) once S(b) has been
    // read (s_free), dQ/dK += dS(b) X(b) once dS is written, then dP(b + 1), which
    // overwrites dS(b) after the product that reads it.
    const uint32_t idesc_s = make_idesc(BF16, 128, kBN, false, false);
    const uint32_t idesc_acc = make_idesc(BF16, 128, C::D, false, true);
    const uint64_t da1 = make_sdesc_sw128(smem_u32(smem + C::kOffA), 16, 1024);
    const uint64_t dx0 = make_sdesc_sw128(smem_u32(smem + C::kOffX), 16, 1024);
    const uint64_t dy0 = make_sdesc_sw128(smem_u32(smem + C::kOffY), 16, 1024);
    // the accumulating product's B operand, MN-major: X (dQ, dK) or Y (dV)
    const uint64_t dacc0 =
        make_sdesc_sw128(smem_u32(smem + (kDV ? C::kOffY : C::kOffX)), C::kBlkBox, 1024);
    constexpr uint32_t kStep = C::kBlkBytes >> 4;
    auto issue_acc = [&](int b) {
      const uint32_t a_col = kDV ? C::kColS + (b & 1) * 64 : C::kColDP;
      const int stage = kDV ? b % NY : b % NX;
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)
        mma_ts(tmem + C::kColAcc, tmem + a_col + kk * 8,
               dacc0 + stage * kStep + ((kk * 2048) >> 4), idesc_acc,
               (b > 0 || kk > 0) ? 1u : 0u);
    };
    auto issue_s = [&](int b) -> bool {
      if (!warp_wait(&x_full[b % NX], (b / NX) & 1, limit, abort_flag, kSiteX)) return false;
      tc_fence_after();
      if (elect_one()) {
        if constexpr (C::kA1Tmem)
          issue_rowdot_ts_wide(tmem + C::kColS + (b % NB) * 64, tmem + C::kColA2,
                               dx0 + (b % NX) * kStep, idesc_s);
        else
          issue_rowdot_wide(tmem + C::kColS + (b % NB) * 64, da1, dx0 + (b % NX) * kStep,
                            idesc_s);
        mma_commit(&s_full[b % NB]);
        if (kDV) mma_commit(&x_empty[b % NX]);  // dV: X is read by S alone
      }
      __syncwarp();
      return true;
    };
    auto issue_dp = [&](int b) -> bool {
      if (!warp_wait(&y_full[b % NY], (b / NY) & 1, limit, abort_flag, kSiteY)) return false;
      tc_fence_after();
      if (elect_one()) {
        issue_rowdot_ts_wide(tmem + C::kColDP, tmem + C::kColA2, dy0 + (b % NY) * kStep,
                             idesc_s);
        mma_commit(dp_full);
        mma_commit(&y_empty[b % NY]);  // dQ/dK: Y is read by dP alone
      }
      __syncwarp();
      return true;
    };
    bool ok = n > 0 && (C::kA1Tmem || warp_wait(a_full, 0, limit, abort_flag, kSiteA));
    if (ok) ok = warp_wait(a2_tmem, 0, limit, abort_flag, kSiteA);
    if (ok) ok = issue_s(0);
    if (ok && C::kA2Tmem) ok = issue_dp(0);
    for (int b = 0; ok && b < n; ++b) {
      if (b + 1 < n) {
        if (C::kA2Tmem &&
            !(ok = warp_wait(s_free, b & 1, limit, abort_flag, kSiteS)))
          break;
        if (!(ok = issue_s(b + 1))) break;
      }
      if constexpr (kDV) {
        if (!(ok = warp_wait(&y_full[b % NY], (b / NY) & 1, limit, abort_flag, kSiteY)))
          break;
      }
      if (!(ok = warp_wait(&ds_full[b % NB], (b / NB) & 1, limit, abort_flag, kSiteDS))) break;
      tc_fence_after();
      if (elect_one()) {
        issue_acc(b);
        mma_commit(kDV ? &y_empty[b % NY] : &x_empty[b % NX]);
        if (b == n - 1) mma_commit(acc_last);
      }
      __syncwarp();
      if (C::kA2Tmem && b + 1 < n && !(ok = issue_dp(b + 1))) break;
    }
    // Every MMA issued must finish before tensor memory is released.
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, kDrainLimit, nullptr, kSiteDrain);
  } else {
    // ------------------------------ elementwise -------------------------------
    const int wq = warp;  // rows [32 wq, 32 wq + 32) of the tile: its tensor-memory lanes
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const int r_in = wq * 32 + lane;
    const int row = r0 + r_in;  // query (dQ) or key (dK, dV) index of this thread
    const float2 sl2x2 = make_float2(p.scale_log2, p.scale_log2);
    // dQ: this row's -L log2(e) and D (rows past N: P = 0). dK/dV: the statistics of the
    // block's 64 queries, staged per block in shared memory by threads 0-63 (-L log2 e)
    // and 64-127 (D), one block ahead in registers.
    float row_nl = -INFINITY, row_d = 0.f;
    if (kRowsAreQueries && row < N) {
      row_nl = -p.lse[sl.stat0 + row] * kLog2e;
      row_d = p.delta[sl.stat0 + row];
    }
    auto load_stat = [&](int b) -> float {
      const int q = (b0 + b) * kBN + (r_in & 63);
      if (q >= N) return r_in < 64 ? -INFINITY : 0.f;  // padding queries: P = 0, D = 0
      return r_in < 64 ? -p.lse[sl.stat0 + q] * kLog2e : p.delta[sl.stat0 + q];
    };
    float stat_next = kRowsAreQueries ? 0.f : load_stat(0);
    if (n > 0) {
      // This row of dO_i (dQ), V_j (dK) or K_j (dV) into tensor memory (rows past the
      // slice's end as zeros): the A operand of dP (dQ, dK) or of S^T (dV).
      const uint8_t* gsrc = reinterpret_cast<const uint8_t*>(
          kRowsAreQueries ? p.in_do : (kDV ? p.in_k : p.in_v));
      const size_t elem0 = kRowsAreQueries ? sl.q_elem0 : sl.k_elem0;
      copy_row_to_tmem<C::D>(row < n_rows ? gsrc + (elem0 + (size_t)row * sl.row_elems) * 2
                                          : nullptr,
                             tmem + lane_base + C::kColA2, p.dh / 8);
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(a2_tmem);
    }
    bool ok = true;
    for (int b = 0; b < n; ++b) {
      const float* st = stats + (b & 1) * 128;
      if constexpr (!kRowsAreQueries) {
        // Buffer b & 1 was last read in block b - 2; every thread has passed block b - 1's
        // stats_ready wait, which needs all four warps' arrivals, so nobody still reads it.
        stats[(b & 1) * 128 + r_in] = stat_next;
        warp_arrive(&stats_ready[b & 1]);
        if (b + 1 < n) stat_next = load_stat(b + 1);
        if (!(ok = warp_wait(&stats_ready[b & 1], (b >> 1) & 1, limit, abort_flag,
                             kWaitDkvStats)))
          break;
      }
      // ---- P = exp2(S * scale * log2(e) - L * log2(e))
      if (!(ok = warp_wait(&s_full[b % NB], (b / NB) & 1, limit, abort_flag, kSiteS))) break;
      tc_fence_after();
      const uint32_t t_s = tmem + lane_base + C::kColS + (b % NB) * 64;
      uint32_t sr[kBN];
      tmem_ld64(t_s, sr);
      if constexpr (C::kA2Tmem) {
        tc_fence_before();
        warp_arrive(s_free);  // S(b) is in registers: S(b + 1) may overwrite it
      }
      float* pr = reinterpret_cast<float*>(sr);
      if constexpr (kRowsAreQueries) {
        const float2 nl = make_float2(row_nl, row_nl);
#pragma unroll
        for (int c = 0; c < kBN; c += 2) {
          const float2 x = fma2(make_float2(pr[c], pr[c + 1]), sl2x2, nl);
          pr[c] = ex2(x.x);
          pr[c + 1] = ex2(x.y);
        }
        const int kbase = b * kBN;  // key of column 0
        if ((p.causal && kbase + kBN - 1 > r0 + off) || kbase + kBN > Nk) {
          int lim = Nk - 1 - kbase;                         // last key in range
          if (p.causal) lim = min(lim, row + off - kbase);  // last key this row sees
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c > lim) pr[c] = 0.f;
        }
      } else {
        const float4* nl4 = reinterpret_cast<const float4*>(st);
#pragma unroll
        for (int c4 = 0; c4 < kBN / 4; ++c4) {
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
        const int qbase = (b0 + b) * kBN;  // query of column 0
        if (p.causal && qbase + off < r0 + kTileM - 1) {
          // query qbase + c sees this key iff qbase + c + off >= row
          const int first = row - off - qbase;
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c < first) pr[c] = 0.f;
        }
      }
      if constexpr (kDV) {
        // P^T as 16-bit pairs over its scores: the A operand of dV += P^T dO
        uint32_t pk[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) pk[u] = pack2<BF16>(pr[2 * u], pr[2 * u + 1]);
        tmem_st16(t_s, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
        tmem_st16(t_s + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
      } else {
        // ---- dS = P * (dP - D), 16-bit pairs over dP: the A operand of the accumulation
        if (!(ok = warp_wait(dp_full, b & 1, limit, abort_flag, kSiteDP))) break;
        tc_fence_after();
        const uint32_t t_dp = tmem + lane_base + C::kColDP;
        uint32_t r[kBN];
        tmem_ld64(t_dp, r);
        if constexpr (kRowsAreQueries) {
          const float2 nd = make_float2(-row_d, -row_d);
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float2 d = mul2(make_float2(pr[2 * u], pr[2 * u + 1]),
                                  add2(make_float2(__uint_as_float(r[2 * u]),
                                                   __uint_as_float(r[2 * u + 1])),
                                       nd));
            r[u] = pack2<BF16>(d.x, d.y);  // in place: r[u] was read in this step or earlier
          }
        } else {
          const float4* dl4 = reinterpret_cast<const float4*>(st + 64);
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
            r[2 * u] = pack2<BF16>(d01.x, d01.y);  // in place, as above
            r[2 * u + 1] = pack2<BF16>(d23.x, d23.y);
          }
        }
        tmem_st16(t_dp, *reinterpret_cast<const uint32_t(*)[16]>(&r[0]));
        tmem_st16(t_dp + 16, *reinterpret_cast<const uint32_t(*)[16]>(&r[16]));
      }
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&ds_full[b % NB]);
    }
    void* out = kRowsAreQueries || MODE == kWideDK ? p.out0 : p.out1;
    const size_t elem0 = kRowsAreQueries ? sl.q_elem0 : sl.k_elem0;
    uint8_t* drow = reinterpret_cast<uint8_t*>(out) + (elem0 + (size_t)row * sl.row_elems) * 2;
    if (n == 0) {
      // keys of a sequence without queries: no query sees them, so their gradients are zero
      uint32_t z[32] = {};
#pragma unroll 1
      for (int cc = 0; cc < C::D / 32; ++cc)
        if (row < n_rows) store_row32<BF16>(drow + cc * 64, z, 1.f, valid16(p.dh, cc * 32, 4));
    } else if (ok && warp_wait(acc_last, 0, limit, abort_flag, kSiteDone)) {
      tc_fence_after();
      const float mul = kDV ? 1.f : p.scale;
#pragma unroll 1
      for (int cc = 0; cc < C::D / 32; ++cc) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + C::kColAcc + cc * 32, a);
        if (row < n_rows) store_row32<BF16>(drow + cc * 64, a, mul, valid16(p.dh, cc * 32, 4));
      }
    }
    tc_fence_before();
  }

  tmem_st_wait();  // no tensor-memory store in flight when memory is released
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// One pass of the kernel above: a1 the resident 128-row tile (dQ, dK), x/y the streamed
// 64-row blocks, a2_rows the tensor whose rows go to tensor memory (dO for dQ, V for dK, K
// for dV); one CTA
// per 128 rows (queries for dQ, keys for dK and dV) of each slice (packed batches: of the
// longest sequence, the tiles past a shorter one's end returning at once).
template <int MODE, bool BF16>
static cudaError_t launch_bwd_wide(const CUtensorMap& a1, const CUtensorMap& x,
                                   const CUtensorMap& y, const void* a2_rows, const Shape& s,
                                   const float* lse, const float* delta, void* out0,
                                   void* out1, cudaStream_t st) {
  using C = BwdWCfg<MODE>;
  auto kern = s.vl.cu_q != nullptr ? attn_bwd_wide_kernel<MODE, BF16, true>
                                   : attn_bwd_wide_kernel<MODE, BF16, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  BwdParams p = {};
  p.in_do = a2_rows;  // dQ: dO, rows copied into tensor memory
  p.in_v = a2_rows;   // dK: V, likewise
  p.in_k = a2_rows;   // dV: K, likewise
  p.lse = lse;
  p.delta = delta;
  p.out0 = out0;
  p.out1 = out1;
  p.dh = s.d;
  p.N = s.N;
  p.Nk = s.Nk;
  p.causal = s.causal ? 1 : 0;
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  p.stall = s.stall;
  p.vl = s.vl;
  const int rows = MODE == kWideDQ ? s.N : s.Nk;  // packed: the longest sequence
  dim3 grid((rows + kTileM - 1) / kTileM, s.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(a1, x, y, p);
  return cudaGetLastError();
}

}  // namespace attn
