// fwd_wide.cuh - the attention forward for head dimensions above 128 (up to 256): the same
// method as fwd.cuh (online softmax over key blocks, exp2 with the scale folded in, P
// rounded to the input type for P V and O divided by the sum of those rounded values, the
// conditional rescale, L = m + ln l) on a tile shape that fits a 256-column head.
//
// Why another shape: at d = 256 one 128-row tile needs 256 tensor-memory columns for O and
// 128 for S, so the two-tile ping-pong of fwd.cuh (768 columns) does not fit in 512, and a
// 128 x 256 K or V block takes 64 KiB of shared memory, so a ring of them beside a 64 KiB
// Q tile leaves no room for a second stage. Here:
//  * one CTA = one 128-row query tile of one (b, h) slice (grid: tiles x slices, the tiles
//    of a head adjacent in launch order and longest first, as in fwd.cuh);
//  * keys come in blocks of 64: S = scale Q K_j^T is a 128 x 64 product (N = 64), K_j and
//    V_j take 32 KiB each. K and V have rings of their own beside Q (64 KiB): three K
//    stages, each free again once its S product is done, and two V stages, free once
//    their P V is done, so the copies of K run two blocks ahead of those of V;
//  * S is double buffered in tensor memory (2 x 64 columns) and O takes 256 columns, so
//    S of block j + 1 runs on the tensor core while the softmax works on block j, and
//    P V of block j (N = 256) follows as soon as P is in tensor memory (written over S as
//    16-bit pairs, like the 128-column kernel);
//  * warps 0-3: softmax, one query row per thread (64 scores a block); warp 4: TMA
//    producer; warp 5: MMA issuer and tensor-memory owner.
// Head dimensions between 136 and 248 run on the same kernel: TMA reads the columns past
// d as zero, so every product sees exact zeros there, and only d columns are stored.
#pragma once

#include "fwd.cuh"
#include "fwd_persistent.cuh"

namespace attn {

struct FwdWCfg {
  static constexpr int D = 256;
  static constexpr int kBN = 64;                       // keys per block
  static constexpr int kChunks = D / kBoxCols;         // 64-column boxes per row: 4
  static constexpr int kQBytes = kChunks * kBoxBytes;  // 128 x 256 tile: 64 KiB
  static constexpr int kKVBox = kBN * 128;             // one [64 rows x 64 cols] box: 8 KiB
  static constexpr int kKVBytes = kChunks * kKVBox;    // 64 x 256 block: 32 KiB
  static constexpr int kKStages = 3, kVStages = 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKVBytes;
  static constexpr int kOffBar = kOffV + kVStages * kKVBytes;
  // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2], p_full[2], o_done,
  // o_last, drain
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 + 2 + 1 + 1 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kSmemBytes > 114 * 1024, "two CTAs could share an SM");
  static constexpr int kThreads = 192;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S buffer b at kColS + 64 b (P over its first 32)
  static constexpr uint32_t kColQ = 128;  // one-tile kernel: Q as 16-bit pairs, 128 columns
  static constexpr uint32_t kColO = 256;  // O: 256 columns
};

template <bool BF16, bool PACKED>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_wide_kernel(const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k64,
                         const __grid_constant__ CUtensorMap map_v64, const FwdParams p) {
  using C = FwdWCfg;
  constexpr int NK = C::kKStages, NV = C::kVStages;
  constexpr int kBN = C::kBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NK;  // the stage's S product is done
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;  // the stage's P V product is done
  uint64_t* s_full = v_empty + NV;  // [2] per S buffer
  uint64_t* p_full = s_full + 2;     // [2] per S buffer: P of the buffer's block is written
  uint64_t* o_done = p_full + 2;     // every P V
  // The last P V alone. When the softmax leaves its last block, two P V products can still
  // be in flight (S(j) is issued before P V(j - 1)), so o_done's parity could name either.
  uint64_t* o_last = o_done + 1;
  uint64_t* drain = o_last + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int bh = blockIdx.y;
  SliceRows sl;
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, sl)) return;
  const int N = sl.nq, Nk = sl.nk, off = sl.off;
  const int nqb = (N + kTileM - 1) / kTileM;
  if (PACKED && (int)blockIdx.x >= nqb) return;  // past this sequence's query tiles
  const int q0 = (nqb - 1 - (int)blockIdx.x) * kTileM;  // longest first within a head
  const int nkb = (Nk + kBN - 1) / kBN;
  // causal: up to the block of the last key the tile's last row sees
  const int n_kv = p.causal ? min(nkb, (q0 + kTileM - 1 + off) / kBN + 1) : nkb;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 4);  // one arrival per softmax warp: its rows of Q are in tensor memory
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);  // one arrival per softmax warp
    }
    mbar_init(o_done, 1);
    mbar_init(o_last, 1);
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

  if (warp == 4 && p.stall) {
    // Failure tests: the producer withholds every copy; the consumers' waits run out.
  } else if (warp == 4) {
    // ------------------------------ TMA producer ------------------------------
    if (elect_one()) {
      tma_prefetch_map(&map_k64);
      tma_prefetch_map(&map_v64);
    }
    __syncwarp();
    // K(j) into stage j % NK once S(j - NK) is done; V(j) into stage j % NV once
    // P V(j - NV) is done (each empty barrier completes once per block of its stage, after
    // a copy issued past its wait). K runs NK - 1 blocks ahead of V.
    int k_issued = 0, v_issued = 0;
    auto load_k = [&](int j) -> bool {
      const int s = j % NK;
      if (j >= NK && !warp_wait(&k_empty[s], ((j / NK) - 1) & 1, limit, abort_flag,
                                kWaitFwdEmpty))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(&k_full[s], C::kKVBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffK + s * C::kKVBytes + c * C::kKVBox, &map_k64,
                                &k_full[s], c * kBoxCols, j * kBN, sl, true);
      }
      __syncwarp();
      k_issued = j + 1;
      return true;
    };
    auto load_v = [&](int j) -> bool {
      const int s = j % NV;
      if (j >= NV && !warp_wait(&v_empty[s], ((j / NV) - 1) & 1, limit, abort_flag,
                                kWaitFwdEmpty))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(&v_full[s], C::kKVBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffV + s * C::kKVBytes + c * C::kKVBox, &map_v64,
                                &v_full[s], c * kBoxCols, j * kBN, sl, true);
      }
      __syncwarp();
      v_issued = j + 1;
      return true;
    };
    bool ok = true;
    for (int j = 0; ok && j < min(NK - 1, n_kv); ++j) ok = load_k(j);
    for (int j = 0; ok && j < n_kv; ++j) {
      if (j + NK - 1 < n_kv) ok = load_k(j + NK - 1);
      if (ok) ok = load_v(j);
    }
    if (*abort_flag) {
      // Let every copy this CTA started land before its shared memory is released.
      for (int j = max(0, k_issued - NK); j < k_issued; ++j)
        mbar_wait(&k_full[j % NK], (j / NK) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
      for (int j = max(0, v_issued - NV); j < v_issued; ++j)
        mbar_wait(&v_full[j % NV], (j / NV) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
    }
  } else if (warp == 5) {
    // ------------------------------ MMA issuer --------------------------------
    // Per block j: S(j + 1) into the other S buffer (its previous P was read by P V(j - 1),
    // issued before it: the tensor core runs them in order), then P(j) V_j once the
    // softmax has written P(j).
    const uint32_t idesc_s = make_idesc(BF16, 128, kBN, false, false);
    const uint32_t idesc_o = make_idesc(BF16, 128, C::D, false, true);
    const uint64_t dk0 = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    // V block: MN-major, 64-column boxes C::kKVBox apart along N, 8-row groups 1 KiB apart
    const uint64_t dv0 = make_sdesc_sw128(smem_u32(smem + C::kOffV), C::kKVBox, 1024);
    constexpr uint32_t kStep = C::kKVBytes >> 4;
    auto issue_s = [&](int j) {  // S = Q K^T with Q from tensor memory
      issue_rowdot_ts_wide(tmem + C::kColS + (j & 1) * 64, tmem + C::kColQ,
                           dk0 + (j % NK) * kStep, idesc_s);
    };
    auto issue_pv = [&](int j) {
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)
        mma_ts(tmem + C::kColO, tmem + C::kColS + (j & 1) * 64 + kk * 8,
               dv0 + (j % NV) * kStep + ((kk * 2048) >> 4), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
    };
    bool ok = warp_wait(q_full, 0, limit, abort_flag, kWaitFwdQ);
    if (ok) ok = warp_wait(&k_full[0], 0, limit, abort_flag, kWaitFwdK);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        issue_s(0);
        mma_commit(&s_full[0]);
        mma_commit(&k_empty[0]);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      const int jn = j + 1;
      if (jn < n_kv) {
        if (!(ok = warp_wait(&k_full[jn % NK], (jn / NK) & 1, limit, abort_flag, kWaitFwdK)))
          break;
        tc_fence_after();
        if (elect_one()) {
          issue_s(jn);
          mma_commit(&s_full[jn & 1]);
          mma_commit(&k_empty[jn % NK]);
        }
        __syncwarp();
      }
      if (!(ok = warp_wait(&v_full[j % NV], (j / NV) & 1, limit, abort_flag, kWaitFwdV))) break;
      if (!(ok = warp_wait(&p_full[j & 1], (j >> 1) & 1, limit, abort_flag, kWaitFwdP))) break;
      tc_fence_after();
      if (elect_one()) {
        issue_pv(j);
        mma_commit(o_done);
        mma_commit(&v_empty[j % NV]);
        if (j == n_kv - 1) mma_commit(o_last);
      }
      __syncwarp();
    }
    // Every MMA issued must finish before tensor memory is released.
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitFwdDrain);
  } else {
    // ------------------------------ softmax -----------------------------------
    const int wq = warp;  // rows [32 wq, 32 wq + 32) of the tile: its tensor-memory lanes
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t t_o = tmem + lane_base + C::kColO;
    const int row = q0 + wq * 32 + lane;  // query index of this thread
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running max of scale*log2(e)*S (possibly stale by <= 8)
    float l = 0.f;        // sum of exp2 values (fp32): defines L
    float lr = 0.f;       // sum of the same values rounded to 16 bits: divides O
    bool ok = true;
    {
      // This thread's row of Q into tensor memory (rows past N as zeros): the A operand of
      // S = Q K^T, read there by every S product without shared-memory traffic.
      const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(p.q) +
                            (sl.q_elem0 + (size_t)row * sl.row_elems) * 2;
      copy_row_to_tmem<C::D>(row < N ? qsrc : nullptr, tmem + lane_base + C::kColQ, p.dh / 8);
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(q_full);
    }
    // O *= alpha in tensor memory, 64 columns at a time (the previous P V must be done).
    auto rescale_o = [&](float alpha) {
#pragma unroll 1
      for (int cc = 0; cc < C::D / 64; ++cc) {
        uint32_t r[64];
        tmem_ld64(t_o + cc * 64, r);
#pragma unroll
        for (int i = 0; i < 64; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st32(t_o + cc * 64, *reinterpret_cast<const uint32_t(*)[32]>(&r[0]));
        tmem_st32(t_o + cc * 64 + 32, *reinterpret_cast<const uint32_t(*)[32]>(&r[32]));
      }
    };
    for (int j = 0; j < n_kv; ++j) {
      const uint32_t t_s = tmem + lane_base + C::kColS + (j & 1) * 64;
      if (!(ok = warp_wait(&s_full[j & 1], (j >> 1) & 1, limit, abort_flag, kWaitFwdS))) break;
      tc_fence_after();
      uint32_t sr[kBN];
      tmem_ld64(t_s, sr);
      float* s = reinterpret_cast<float*>(sr);
      const int kbase = j * kBN;
      const bool diag = p.causal && (kbase + kBN - 1 > q0 + off);
      if (diag || kbase + kBN > Nk) {
        int lim = Nk - 1 - kbase;                           // last key in range
        if (p.causal) lim = min(lim, row + off - kbase);    // last key this row sees
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      float mx[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) mx[u] = fmaxf(s[2 * u], s[2 * u + 1]);
#pragma unroll
      for (int c = 8; c < kBN; c += 8) {
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
      float2 sum[4];
      float rsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int u = 0; u < 4; ++u) sum[u] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c2 = 0; c2 < kBN / 32; ++c2) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x =
              fma2(make_float2(s[c2 * 32 + 2 * i], s[c2 * 32 + 2 * i + 1]), sl2x2, neg_m2);
          const float2 pp = make_float2(ex2(x.x), ex2(x.y));
          sum[i & 3] = add2(sum[i & 3], pp);
          pk[i] = pack2<BF16>(pp.x, pp.y);
          add_pair16<BF16>(rsum[(i & 1) * 2], rsum[(i & 1) * 2 + 1], pk[i]);
        }
        tmem_st16(t_s + c2 * 16, pk);  // P over the scores already read
      }
      const float2 sa = add2(add2(sum[0], sum[1]), add2(sum[2], sum[3]));
      l = l * alpha + (sa.x + sa.y);
      lr = lr * alpha + ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3]));
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // Bring O to the new max once P V(j - 1) has landed. o_done is at most one phase
        // past that product here: S(j) was committed after P V(j - 2).
        if (!(ok = warp_wait(o_done, (j - 1) & 1, limit, abort_flag, kWaitFwdO))) break;
        tc_fence_after();
        rescale_o(alpha);
      }
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&p_full[j & 1]);
    }
    if (ok && warp_wait(o_last, 0, limit, abort_flag, kWaitFwdO)) {
      tc_fence_after();
      const float inv_l = 1.f / lr;
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                      (sl.q_elem0 + (size_t)row * sl.row_elems) * 2;
#pragma unroll 1
      for (int cc = 0; cc < C::D / 64; ++cc) {
        uint32_t r[64];
        tmem_ld64(t_o + cc * 64, r);
        if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 128);
          const int n16 = valid16(p.dh, cc * 64, 8);  // columns past dh are not stored
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              w4[i] = pack2<BF16>(__uint_as_float(r[8 * v + 2 * i]) * inv_l,
                                  __uint_as_float(r[8 * v + 2 * i + 1]) * inv_l);
            if (v < n16) dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      if (row < N) p.lse[sl.stat0 + row] = (m + log2f(l)) * kLn2;
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

// ---------------------------------------------------------------------------------------
// The same forward as a persistent kernel: one CTA per SM walks a list of items (128 query
// rows of one (b, h) slice each), so the fixed cost of a CTA (launch, barriers, tensor
// memory, the first copies, the last products, the epilogue) is paid once per SM instead of
// once per tile. The K and V rings, the two S buffers and every barrier phase run on across
// items (running counts kept alike by all roles); each item's first two K blocks are copied
// before its Q, which waits for the previous item's last S product; the first P V of an
// item waits until the previous item's epilogue has read O (o_free). The arithmetic of
// every item is that of the kernel above: the outputs are bit-identical.

struct FwdWPCfg : FwdWCfg {
  // the barriers of the one-tile kernel, then q_empty, o_free, q_tmem_full and q_smem_free
  static constexpr int kNumBarsP = kNumBars + 4;
  static constexpr int kOffMiscP = kOffBar + kNumBarsP * 8;
  static constexpr int kSmemBytesP = kOffMiscP + 16 + 1024;
  static_assert(kSmemBytesP <= 227 * 1024, "shared memory");
};

// One work item of the persistent kernel.
struct FwdWItem {
  SliceRows sl;
  int N, Nk, off;
  int q0;   // first query row of the tile within its slice
  int n;    // key blocks (64 keys each) the tile sees
};

// Geometry of item `item` (nqb_max tiles per slice, longest first within a slice). False:
// nothing to do (a tile past its sequence's end, or a malformed sequence).
template <bool PACKED>
__device__ __forceinline__ bool fwd_wide_item_geom(const FwdParams& p, int item, int nqb_max,
                                                   FwdWItem& it) {
  const int bh = item / nqb_max;
  const int x = item - bh * nqb_max;
  if (!slice_rows<PACKED>(p.vl, bh, p.N, p.Nk, p.dh, p.causal != 0, it.sl)) return false;
  it.N = it.sl.nq;
  it.Nk = it.sl.nk;
  it.off = it.sl.off;
  const int nqb = (it.N + kTileM - 1) / kTileM;
  if (x >= nqb) return false;
  it.q0 = (nqb - 1 - x) * kTileM;
  const int nkb = (it.Nk + FwdWCfg::kBN - 1) / FwdWCfg::kBN;
  it.n = p.causal ? min(nkb, (it.q0 + kTileM - 1 + it.off) / FwdWCfg::kBN + 1) : nkb;
  return it.n > 0;
}

template <bool BF16, bool PACKED, class Sched>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_wide_persistent_kernel(const __grid_constant__ CUtensorMap map_q,
                                    const __grid_constant__ CUtensorMap map_k64,
                                    const __grid_constant__ CUtensorMap map_v64,
                                    const FwdParams p, int n_items, int nqb_max,
                                    const __grid_constant__ Sched sched) {
  using C = FwdWPCfg;
  constexpr int NK = C::kKStages, NV = C::kVStages;
  constexpr int kBN = C::kBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;  // [2] per S buffer
  uint64_t* p_full = s_full + 2;    // [2] per S buffer
  uint64_t* o_done = p_full + 2;    // every P V
  uint64_t* o_last = o_done + 1;    // the last P V of an item
  uint64_t* drain = o_last + 1;
  uint64_t* q_empty = drain + 1;    // every S of the item is done: Q may be replaced
  uint64_t* o_free = q_empty + 1;   // the epilogue has read O
  // Q goes HBM -> shared memory (TMA, q_full) -> tensor memory (the softmax threads, a row
  // each: q_tmem_full), where it is the A operand of every S of the item; the shared tile is
  // then free for the next item's copy (q_smem_free).
  uint64_t* q_tmem_full = o_free + 1;
  uint64_t* q_smem_free = q_tmem_full + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMiscP);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMiscP + 4);

  const int warp = warp_id();
  const int lane = lane_id();
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
    }
    mbar_init(o_done, 1);
    mbar_init(o_last, 1);
    mbar_init(drain, 1);
    mbar_init(q_empty, 1);
    mbar_init(o_free, 4);  // one arrival per softmax warp
    mbar_init(q_tmem_full, 4);
    mbar_init(q_smem_free, 4);
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

  if (warp == 4 && p.stall) {
    // Failure tests: the producer withholds every copy; the consumers' waits run out.
  } else if (warp == 4) {
    // ------------------------------ TMA producer ------------------------------
    if (elect_one()) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k64);
      tma_prefetch_map(&map_v64);
    }
    __syncwarp();
    // Running counts of the copies issued: K and V blocks (one count per block of every
    // item, in item order), Q tiles.
    int k_issued = 0, v_issued = 0, q_loads = 0;
    bool ok = true;
    auto load_k = [&](const FwdWItem& it, int gb, int j) -> bool {
      const int s = gb % NK;
      if (gb >= NK &&
          !warp_wait(&k_empty[s], ((gb / NK) - 1) & 1, limit, abort_flag, kWaitFwdEmpty))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(&k_full[s], C::kKVBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffK + s * C::kKVBytes + c * C::kKVBox, &map_k64,
                                &k_full[s], c * kBoxCols, j * kBN, it.sl, true);
      }
      __syncwarp();
      k_issued = gb + 1;
      return true;
    };
    auto load_v = [&](const FwdWItem& it, int gb, int j) -> bool {
      const int s = gb % NV;
      if (gb >= NV &&
          !warp_wait(&v_empty[s], ((gb / NV) - 1) & 1, limit, abort_flag, kWaitFwdEmpty))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(&v_full[s], C::kKVBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffV + s * C::kKVBytes + c * C::kKVBox, &map_v64,
                                &v_full[s], c * kBoxCols, j * kBN, it.sl, true);
      }
      __syncwarp();
      v_issued = gb + 1;
      return true;
    };
    for (int k = 0; ok; ++k) {
      const int item = fwd_sched_item(sched, k, G, cta, n_items);
      if (item < 0) break;
      FwdWItem it;
      if (!fwd_wide_item_geom<PACKED>(p, item, nqb_max, it)) continue;
      const int gb0 = v_issued;  // global index of the item's first block
      constexpr int kLead = NK - 1;
      for (int j = 0; ok && j < min(kLead, it.n); ++j) ok = load_k(it, gb0 + j, j);
      if (!ok) break;
      // The softmax threads must have copied the previous item's Q out of shared memory
      // (q_smem_free completes once per item; its next completion needs the Q copied below).
      if (q_loads > 0 &&
          !(ok = warp_wait(q_smem_free, (q_loads - 1) & 1, limit, abort_flag, kWaitFwdQEmpty)))
        break;
      if (elect_one()) {
        mbar_arrive_expect_tx(q_full, C::kQBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_rows<PACKED>(smem + C::kOffQ + c * kBoxBytes, &map_q, q_full, c * kBoxCols,
                                it.q0, it.sl, false);
      }
      __syncwarp();
      ++q_loads;
      for (int j = 0; ok && j < it.n; ++j) {
        if (j + kLead < it.n) ok = load_k(it, gb0 + j + kLead, j + kLead);
        if (ok) ok = load_v(it, gb0 + j, j);
      }
    }
    if (*abort_flag) {
      // Let every copy this CTA started land before its shared memory is released.
      if (q_loads > 0) mbar_wait(q_full, (q_loads - 1) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
      for (int b = max(0, k_issued - NK); b < k_issued; ++b)
        mbar_wait(&k_full[b % NK], (b / NK) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
      for (int b = max(0, v_issued - NV); b < v_issued; ++b)
        mbar_wait(&v_full[b % NV], (b / NV) & 1, kDrainLimit, nullptr, kWaitFwdDrain);
    }
  } else if (warp == 5) {
    // ------------------------------ MMA issuer --------------------------------
    const uint32_t idesc_s = make_idesc(BF16, 128, kBN, false, false);
    const uint32_t idesc_o = make_idesc(BF16, 128, C::D, false, true);
    const uint64_t dk0 = make_sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dv0 = make_sdesc_sw128(smem_u32(smem + C::kOffV), C::kKVBox, 1024);
    constexpr uint32_t kStep = C::kKVBytes >> 4;
    // S(b) = Q K^T into buffer b & 1, Q from tensor memory (its previous contents, P(b - 2),
    // were read by P V(b - 2), issued before: the tensor core runs them in order)
    auto issue_s = [&](int b) -> bool {
      if (!warp_wait(&k_full[b % NK], (b / NK) & 1, limit, abort_flag, kWaitFwdK)) return false;
      tc_fence_after();
      if (elect_one()) {
        issue_rowdot_ts_wide(tmem + C::kColS + (b & 1) * 64, tmem + C::kColQ,
                             dk0 + (b % NK) * kStep, idesc_s);
        mma_commit(&s_full[b & 1]);
        mma_commit(&k_empty[b % NK]);
      }
      __syncwarp();
      return true;
    };
    int gb = 0, items = 0;  // running counts: blocks and items
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = fwd_sched_item(sched, k, G, cta, n_items);
      if (item < 0) break;
      FwdWItem it;
      if (!fwd_wide_item_geom<PACKED>(p, item, nqb_max, it)) continue;
      const int n = it.n;
      if (!(ok = warp_wait(q_tmem_full, items & 1, limit, abort_flag, kWaitFwdQ))) break;
      if (!(ok = issue_s(gb))) break;
      if (n == 1) {
        if (elect_one()) mma_commit(q_empty);  // every S of the item issued
        __syncwarp();
      }
      for (int j = 0; ok && j < n; ++j) {
        const int b = gb + j;
        if (j + 1 < n) {
          if (!(ok = issue_s(b + 1))) break;
          if (j + 2 == n) {
            if (elect_one()) mma_commit(q_empty);
            __syncwarp();
          }
        }
        if (!(ok = warp_wait(&v_full[b % NV], (b / NV) & 1, limit, abort_flag, kWaitFwdV)))
          break;
        if (!(ok = warp_wait(&p_full[b & 1], (b >> 1) & 1, limit, abort_flag, kWaitFwdP)))
          break;
        // The item's first P V overwrites O: the previous item's epilogue must have read it
        // (o_free: one completion per item, each after an o_last that follows this wait).
        if (j == 0 && items > 0 &&
            !(ok = warp_wait(o_free, (items - 1) & 1, limit, abort_flag, kWaitFwdOFree)))
          break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts(tmem + C::kColO, tmem + C::kColS + (b & 1) * 64 + kk * 8,
                   dv0 + (b % NV) * kStep + ((kk * 2048) >> 4), idesc_o,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(o_done);
          mma_commit(&v_empty[b % NV]);
          if (j == n - 1) mma_commit(o_last);
        }
        __syncwarp();
      }
      gb += n;
      ++items;
    }
    // Every MMA issued must finish before tensor memory is released.
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, kDrainLimit, nullptr, kWaitFwdDrain);
  } else {
    // ------------------------------ softmax -----------------------------------
    const int wq = warp;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t t_o = tmem + lane_base + C::kColO;
    const float sl2 = p.scale_log2;
    auto rescale_o = [&](float alpha) {
#pragma unroll 1
      for (int cc = 0; cc < C::D / 64; ++cc) {
        uint32_t r[64];
        tmem_ld64(t_o + cc * 64, r);
#pragma unroll
        for (int i = 0; i < 64; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st32(t_o + cc * 64, *reinterpret_cast<const uint32_t(*)[32]>(&r[0]));
        tmem_st32(t_o + cc * 64 + 32, *reinterpret_cast<const uint32_t(*)[32]>(&r[32]));
      }
    };
    int gb = 0, items = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int item = fwd_sched_item(sched, k, G, cta, n_items);
      if (item < 0) break;
      FwdWItem it;
      if (!fwd_wide_item_geom<PACKED>(p, item, nqb_max, it)) continue;
      const int row = it.q0 + wq * 32 + lane;  // query index of this thread
      float m = -INFINITY, l = 0.f, lr = 0.f;
      {
        // This thread's row of the item's Q: from the shared tile (four 128-byte-swizzled
        // boxes of 64 columns) into tensor memory, once the previous item's S products are
        // done with the tensor-memory copy (q_empty); then both copies are signalled.
        if (!(ok = warp_wait(q_full, items & 1, limit, abort_flag, kWaitFwdQ))) break;
        if (items > 0 &&
            !(ok = warp_wait(q_empty, (items - 1) & 1, limit, abort_flag, kWaitFwdQEmpty)))
          break;
        tc_fence_after();
        const int r_in = wq * 32 + lane;
        const uint8_t* qrow = smem + C::kOffQ + r_in * 128;
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(qrow + c * kBoxBytes +
                                                           ((j ^ (r_in & 7)) << 4));
            r[4 * j] = v.x;
            r[4 * j + 1] = v.y;
            r[4 * j + 2] = v.z;
            r[4 * j + 3] = v.w;
          }
          tmem_st32(tmem + lane_base + C::kColQ + c * 32, r);
        }
        tmem_st_wait();
        tc_fence_before();
        fence_proxy_async_smem();  // the reads above before the next TMA copy into the tile
        warp_arrive(q_tmem_full);
        warp_arrive(q_smem_free);
      }
      for (int j = 0; j < it.n; ++j) {
        const int b = gb + j;
        const uint32_t t_s = tmem + lane_base + C::kColS + (b & 1) * 64;
        if (!(ok = warp_wait(&s_full[b & 1], (b >> 1) & 1, limit, abort_flag, kWaitFwdS)))
          break;
        tc_fence_after();
        uint32_t sr[kBN];
        tmem_ld64(t_s, sr);
        float* s = reinterpret_cast<float*>(sr);
        const int kbase = j * kBN;
        const bool diag = p.causal && (kbase + kBN - 1 > it.q0 + it.off);
        if (diag || kbase + kBN > it.Nk) {
          int lim = it.Nk - 1 - kbase;
          if (p.causal) lim = min(lim, row + it.off - kbase);
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
        float mx[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) mx[u] = fmaxf(s[2 * u], s[2 * u + 1]);
#pragma unroll
        for (int c = 8; c < kBN; c += 8) {
#pragma unroll
          for (int u = 0; u < 4; ++u) mx[u] = fmax3(mx[u], s[c + 2 * u], s[c + 2 * u + 1]);
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
        for (int c2 = 0; c2 < kBN / 32; ++c2) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x =
                fma2(make_float2(s[c2 * 32 + 2 * i], s[c2 * 32 + 2 * i + 1]), sl2x2, neg_m2);
            const float2 pp = make_float2(ex2(x.x), ex2(x.y));
            sum[i & 3] = add2(sum[i & 3], pp);
            pk[i] = pack2<BF16>(pp.x, pp.y);
            add_pair16<BF16>(rsum[(i & 1) * 2], rsum[(i & 1) * 2 + 1], pk[i]);
          }
          tmem_st16(t_s + c2 * 16, pk);
        }
        const float2 sa = add2(add2(sum[0], sum[1]), add2(sum[2], sum[3]));
        l = l * alpha + (sa.x + sa.y);
        lr = lr * alpha + ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3]));
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // o_done is at most one phase past P V(b - 1) here: S(b) was committed after
          // P V(b - 2).
          if (!(ok = warp_wait(o_done, (b - 1) & 1, limit, abort_flag, kWaitFwdO))) break;
          tc_fence_after();
          rescale_o(alpha);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&p_full[b & 1]);
      }
      if (!ok) break;
      // Epilogue: O in four 64-column pieces, each normalised and stored as it is read;
      // O is released (o_free) after the last read.
      if (!(ok = warp_wait(o_last, items & 1, limit, abort_flag, kWaitFwdO))) break;
      tc_fence_after();
      const float inv_l = 1.f / lr;
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                      (it.sl.q_elem0 + (size_t)row * it.sl.row_elems) * 2;
#pragma unroll 1
      for (int cc = 0; cc < C::D / 64; ++cc) {
        uint32_t r[64];
        tmem_ld64(t_o + cc * 64, r);
        if (cc == C::D / 64 - 1) {
          tc_fence_before();
          warp_arrive(o_free);
        }
        if (row < it.N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 128);
          const int n16 = valid16(p.dh, cc * 64, 8);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              w4[i] = pack2<BF16>(__uint_as_float(r[8 * v + 2 * i]) * inv_l,
                                  __uint_as_float(r[8 * v + 2 * i + 1]) * inv_l);
            if (v < n16) dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      if (row < it.N) p.lse[it.sl.stat0 + row] = (m + log2f(l)) * kLn2;
      gb += it.n;
      ++items;
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

}  // namespace attn
