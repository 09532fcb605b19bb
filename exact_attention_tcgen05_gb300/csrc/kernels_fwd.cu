// kernels_fwd.cu - instantiation and launch of the forward kernel.
#include <algorithm>
#include <cstdlib>
#include <vector>

#include "fwd.cuh"
#include "fwd_pair.cuh"
#include "fwd_persistent.cuh"
#include "fwd_wide.cuh"
#include "launch.h"

namespace attn {

static int sm_count_fwd() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

// Which forward: the persistent kernel (fwd_persistent.cuh) except at d = 64 with long
// items (24 or more key blocks per item on average), where the one-item kernel's loop
// measured about 5% faster and the fixed cost per item matters little. Head dims above 128
// (fwd_wide.cuh, 64-key blocks): the persistent kernel for causal items of fewer than 96
// key blocks on average and other items of fewer than 48 (measured on GB300, d = 256:
// causal B16 H16 N1024 0.200 -> 0.163 ms, B4 H16 N4096 0.432 -> 0.399 ms, B2 H16 N8192
// 0.744 -> 0.724 ms), the one-tile kernel for longer ones (B4 H16 N4096 full 0.720
// against 0.730 ms, B1 H16 N16384 causal 1.35 against 1.39 ms).
// ATTN_FWD_PERSISTENT = 0 / 1 forces one or the other (both give the same bits).
static bool use_persistent_fwd(const Shape& s) {
  static const int forced = [] {
    const char* e = std::getenv("ATTN_FWD_PERSISTENT");
    return e == nullptr ? -1 : (e[0] == '0' ? 0 : 1);
  }();
  if (forced >= 0) return forced == 1;
  if (s.d > 128) {
    const int nkb64 = (s.Nk + 63) / 64;
    return s.causal ? (nkb64 + 1) / 2 < 96 : nkb64 < 48;
  }
  const int nkb = (s.Nk + kTileN - 1) / kTileN;
  const int blocks_per_item = s.causal ? (nkb + 1) / 2 : nkb;
  return !(s.d <= 64 && blocks_per_item >= 24);
}

// Key blocks item slot `x` of a slice with nq queries and nk keys works through (the larger
// of its two tiles; the same geometry as fwd_item_geom); 0 past the slice's end.
static int fwd_item_blocks(int nq, int nk, bool causal, int x) {
  const int nqb = (nq + 2 * kTileM - 1) / (2 * kTileM);
  if (x >= nqb) return 0;
  const int nkb = (nk + kTileN - 1) / kTileN;
  const int off = nk - nq;
  const int q0 = (nqb - 1 - x) * 2 * kTileM;
  const int ntiles = (q0 + kTileM < nq) ? 2 : 1;
  int n = 0;
  for (int t = 0; t < ntiles; ++t)
    n = std::max(n, causal ? std::min(nkb, (q0 + t * kTileM + kTileM - 1 + off) / kTileN + 1)
                           : nkb);
  return n;
}

// The persistent forward's table (schedule.h) for causal dense inputs, or packed batches
// whose host lengths are known, with more items than CTAs: cost = key blocks + 1 for an
// item's fixed cost, windows of heads by their K/V bytes. False: the serpentine runs.
static bool fwd_schedule(const Shape& s, int nqb, int G, ItemTable& out) {
  const bool packed = s.vl.cu_q != nullptr;
  const long long n_items = (long long)nqb * s.BH;
  if (!item_table_applies(s.causal, packed, s.host_cu_q != nullptr, n_items, G)) return false;
  static ItemTableCache cache;
  const long long k[8] = {s.BH, s.N, s.Nk, s.d, G, nqb, s.causal ? 1 : 0,
                          lengths_hash(s.host_cu_q, s.host_cu_k, s.vl_b)};
  cache.get(k, G, n_items, out, [&](ItemTable& t) {
    const long long kv_bytes =
        packed ? 4LL * std::max(1, s.vl.total_k / std::max(1, s.vl_b)) * s.d : 4LL * s.Nk * s.d;
    auto cost = [&](int bh, int x) -> long long {
      int nq, nk;
      slice_lengths(s, bh, nq, nk);
      const int n = fwd_item_blocks(nq, nk, s.causal, x);
      return n > 0 ? n + 1 : 0;
    };
    greedy_item_table(s.BH, nqb, cost, item_table_window(s.BH, kv_bytes), G, t);
  });
  return true;
}

// The CTA-pair forward (fwd_pair.cuh) runs only when ATTN_FWD_PAIR = 1, in place of the
// 128-column persistent forward; it gives the same bits. Measured on GB300 it is slower
// (B4 H32 N4096 causal: 0.574 against 0.420 ms): the forward is bound by each tile's chain
// S -> softmax -> P V, not by its copies or products, and the pair adds the wait for the
// other CTA's P to that chain.
static bool use_pair_fwd(const Shape& s) {
  static const bool on = [] {
    const char* e = std::getenv("ATTN_FWD_PAIR");
    return e != nullptr && e[0] == '1';
  }();
  return on && s.d > 64 && use_persistent_fwd(s);
}

// Key blocks of pair item slot `x` (512 query rows; the geometry of fwd_pair_item_geom).
static int fwd_pair_item_blocks(int nq, int nk, bool causal, int x) {
  const int nsb = (nq + 4 * kTileM - 1) / (4 * kTileM);
  if (x >= nsb) return 0;
  const int nkb = (nk + kTileN - 1) / kTileN;
  const int off = nk - nq;
  const int q0 = (nsb - 1 - x) * 4 * kTileM;
  int n = 0;
  for (int t = 0; t < 2; ++t) {
    const int r0 = q0 + t * 2 * kTileM;
    if (r0 >= nq) continue;
    const int last = std::min(r0 + 2 * kTileM, nq) - 1;
    n = std::max(n, causal ? std::min(nkb, (last + off) / kTileN + 1) : nkb);
  }
  return n;
}

static bool fwd_pair_schedule(const Shape& s, int nsb, int G, ItemTable& out) {
  const bool packed = s.vl.cu_q != nullptr;
  const long long n_items = (long long)nsb * s.BH;
  if (!item_table_applies(s.causal, packed, s.host_cu_q != nullptr, n_items, G)) return false;
  static ItemTableCache cache;
  const long long k[8] = {s.BH, s.N, s.Nk, s.d, G, nsb, s.causal ? 1 : 0,
                          lengths_hash(s.host_cu_q, s.host_cu_k, s.vl_b)};
  cache.get(k, G, n_items, out, [&](ItemTable& t) {
    const long long kv_bytes =
        packed ? 4LL * std::max(1, s.vl.total_k / std::max(1, s.vl_b)) * s.d : 4LL * s.Nk * s.d;
    auto cost = [&](int bh, int x) -> long long {
      int nq, nk;
      slice_lengths(s, bh, nq, nk);
      const int n = fwd_pair_item_blocks(nq, nk, s.causal, x);
      return n > 0 ? n + 1 : 0;
    };
    greedy_item_table(s.BH, nsb, cost, item_table_window(s.BH, kv_bytes), G, t);
  });
  return true;
}

// Clusters of two CTAs of `kern` (320 threads, `smem` bytes each) that fit on the device at
// once, asked of the runtime once per device: the persistent pair grid's size.
template <class Kern>
static int pair_clusters(Kern kern, int smem) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return sm_count_fwd() / 2;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count_fwd() / 2), 1, 1);
  cfg.blockDim = dim3(320, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sm_count_fwd() / 2;
  }
  n = std::min(n, kItemTableMaxCtas);
  cached[dev] = n;
  return n;
}

template <bool BF16, bool PACKED>
static cudaError_t launch_fwd_pair(const Maps& m, const Shape& s, const FwdParams& p,
                                   cudaStream_t st) {
  using CP = FwdPairCfg<128>;
  const int nsb_max = (s.N + 4 * kTileM - 1) / (4 * kTileM);
  const long long n_items = (long long)nsb_max * s.BH;
  auto kt = attn_fwd_pair_kernel<BF16, PACKED, ItemTable>;
  auto ks = attn_fwd_pair_kernel<BF16, PACKED, FwdSerpentine>;
  cudaError_t e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       CP::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, CP::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int G = (int)std::min<long long>(n_items, pair_clusters(ks, CP::kSmemBytes));
  static thread_local ItemTable table;
  if (fwd_pair_schedule(s, nsb_max, G, table))
    kt<<<2 * G, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k64, m.v, p, (int)n_items, nsb_max,
                                                    table);
  else
    ks<<<2 * G, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k64, m.v, p, (int)n_items, nsb_max,
                                                    FwdSerpentine{});
  return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_fwd_t(const Maps& m, const Shape& s, void* o, float* lse,
                                cudaStream_t st) {
  using C = FwdCfg<D>;
  auto kern = s.vl.cu_q != nullptr ? attn_fwd_kernel<D, BF16, true>
                                   : attn_fwd_kernel<D, BF16, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.q = nullptr;
  p.o = o;
  p.lse = lse;
  p.dh = s.d;
  p.N = s.N;
  p.Nk = s.Nk;
  p.causal = s.causal ? 1 : 0;
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  p.stall = s.stall;
  p.vl = s.vl;
  // Packed batches: s.N is the longest query sequence; blocks past a sequence's end are
  // skipped.
  const int nqb_max = (s.N + 2 * kTileM - 1) / (2 * kTileM);
  if constexpr (D == 128) {
    if (use_pair_fwd(s))
      return s.vl.cu_q != nullptr ? launch_fwd_pair<BF16, true>(m, s, p, st)
                                  : launch_fwd_pair<BF16, false>(m, s, p, st);
  }
  if (use_persistent_fwd(s)) {
    using CP = FwdPCfg<D>;
    const long long n_items = (long long)nqb_max * s.BH;
    const int grid = (int)std::min<long long>(n_items, sm_count_fwd());
    static thread_local ItemTable table;  // 29 KiB: not on the stack
    if (fwd_schedule(s, nqb_max, grid, table)) {
      auto kt = s.vl.cu_q != nullptr ? attn_fwd_persistent_kernel<D, BF16, true, ItemTable>
                                     : attn_fwd_persistent_kernel<D, BF16, false, ItemTable>;
      e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, CP::kSmemBytes);
      if (e != cudaSuccess) return e;
      kt<<<grid, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k, m.v, m.o, p, (int)n_items,
                                                     nqb_max, table);
      return cudaGetLastError();
    }
    auto kp = s.vl.cu_q != nullptr ? attn_fwd_persistent_kernel<D, BF16, true, FwdSerpentine>
                                   : attn_fwd_persistent_kernel<D, BF16, false, FwdSerpentine>;
    e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, CP::kSmemBytes);
    if (e != cudaSuccess) return e;
    kp<<<grid, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k, m.v, m.o, p, (int)n_items,
                                                   nqb_max, FwdSerpentine{});
    return cudaGetLastError();
  }
  dim3 grid(nqb_max, s.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(m.q, m.k, m.v, p);
  return cudaGetLastError();
}

// Key blocks (64 keys) tile slot `x` of a slice with nq queries and nk keys sees in the
// 256-column forward (the geometry of fwd_wide_item_geom); 0 past the slice's end.
static int fwd_wide_item_blocks(int nq, int nk, bool causal, int x) {
  const int nqb = (nq + kTileM - 1) / kTileM;
  if (x >= nqb) return 0;
  const int nkb = (nk + FwdWCfg::kBN - 1) / FwdWCfg::kBN;
  const int q0 = (nqb - 1 - x) * kTileM;
  return causal ? std::min(nkb, (q0 + kTileM - 1 + nk - nq) / FwdWCfg::kBN + 1) : nkb;
}

// The persistent 256-column forward's table (schedule.h), as for the 128-column one.
static bool fwd_wide_schedule(const Shape& s, int nqb, int G, ItemTable& out) {
  const bool packed = s.vl.cu_q != nullptr;
  const long long n_items = (long long)nqb * s.BH;
  if (!item_table_applies(s.causal, packed, s.host_cu_q != nullptr, n_items, G)) return false;
  static ItemTableCache cache;
  const long long k[8] = {s.BH, s.N, s.Nk, s.d, G, nqb, s.causal ? 1 : 0,
                          lengths_hash(s.host_cu_q, s.host_cu_k, s.vl_b)};
  cache.get(k, G, n_items, out, [&](ItemTable& t) {
    const long long kv_bytes =
        packed ? 4LL * std::max(1, s.vl.total_k / std::max(1, s.vl_b)) * s.d : 4LL * s.Nk * s.d;
    auto cost = [&](int bh, int x) -> long long {
      int nq, nk;
      slice_lengths(s, bh, nq, nk);
      const int n = fwd_wide_item_blocks(nq, nk, s.causal, x);
      return n > 0 ? n + 1 : 0;
    };
    greedy_item_table(s.BH, nqb, cost, item_table_window(s.BH, kv_bytes), G, t);
  });
  return true;
}

// Head dims above 128: the 256-column forward (fwd_wide.cuh): the persistent kernel, or
// with ATTN_FWD_PERSISTENT = 0 one CTA per 128-row tile (the same bits).
template <bool BF16>
static cudaError_t launch_fwd_wide(const Maps& m, const Shape& s, const void* q, void* o,
                                   float* lse, cudaStream_t st) {
  using C = FwdWCfg;
  auto kern = s.vl.cu_q != nullptr ? attn_fwd_wide_kernel<BF16, true>
                                   : attn_fwd_wide_kernel<BF16, false>;
  cudaError_t e;
  FwdParams p;
  p.q = q;
  p.o = o;
  p.lse = lse;
  p.dh = s.d;
  p.N = s.N;
  p.Nk = s.Nk;
  p.causal = s.causal ? 1 : 0;
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  p.stall = s.stall;
  p.vl = s.vl;
  const int nqb_max = (s.N + kTileM - 1) / kTileM;
  if (use_persistent_fwd(s)) {
    using CP = FwdWPCfg;
    const long long n_items = (long long)nqb_max * s.BH;
    const int grid = (int)std::min<long long>(n_items, sm_count_fwd());
    static thread_local ItemTable table;
    if (fwd_wide_schedule(s, nqb_max, grid, table)) {
      auto kt = s.vl.cu_q != nullptr ? attn_fwd_wide_persistent_kernel<BF16, true, ItemTable>
                                     : attn_fwd_wide_persistent_kernel<BF16, false, ItemTable>;
      e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               CP::kSmemBytesP);
      if (e != cudaSuccess) return e;
      kt<<<grid, CP::kThreads, CP::kSmemBytesP, st>>>(m.q, m.k64, m.v64, p, (int)n_items,
                                                      nqb_max, table);
      return cudaGetLastError();
    }
    auto ks = s.vl.cu_q != nullptr ? attn_fwd_wide_persistent_kernel<BF16, true, FwdSerpentine>
                                   : attn_fwd_wide_persistent_kernel<BF16, false, FwdSerpentine>;
    e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, CP::kSmemBytesP);
    if (e != cudaSuccess) return e;
    ks<<<grid, CP::kThreads, CP::kSmemBytesP, st>>>(m.q, m.k64, m.v64, p, (int)n_items,
                                                    nqb_max, FwdSerpentine{});
    return cudaGetLastError();
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(nqb_max, s.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(m.q, m.k64, m.v64, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const Maps& m, const Shape& s, const void* q, void* o, float* lse,
                       cudaStream_t st) {
  if (s.d > 128) return s.bf16 ? launch_fwd_wide<true>(m, s, q, o, lse, st)
                                : launch_fwd_wide<false>(m, s, q, o, lse, st);
  if (s.d > 64) return s.bf16 ? launch_fwd_t<128, true>(m, s, o, lse, st)
                                : launch_fwd_t<128, false>(m, s, o, lse, st);
  return s.bf16 ? launch_fwd_t<64, true>(m, s, o, lse, st)
                : launch_fwd_t<64, false>(m, s, o, lse, st);
}

ATTN_DEFINE_STATUS_READER(status_fwd)

}  // namespace attn
