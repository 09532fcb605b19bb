// kernels_fwd.cu - instantiation and launch of the forward kernel.
#include <algorithm>
#include <cstdlib>
#include <vector>

#include "fwd.cuh"
#include "fwd_persistent.cuh"
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
// measured about 5% faster and the fixed cost per item matters little. ATTN_FWD_PERSISTENT
// = 0 / 1 forces one or the other (both give the same bits).
static bool use_persistent_fwd(const Shape& s) {
  static const int forced = [] {
    const char* e = std::getenv("ATTN_FWD_PERSISTENT");
    return e == nullptr ? -1 : (e[0] == '0' ? 0 : 1);
  }();
  if (forced >= 0) return forced == 1;
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
  p.o = o;
  p.lse = lse;
  p.dh = s.d;
  p.N = s.N;
  p.Nk = s.Nk;
  p.causal = s.causal ? 1 : 0;
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  p.vl = s.vl;
  // Packed batches: s.N is the longest query sequence; blocks past a sequence's end are
  // skipped.
  const int nqb_max = (s.N + 2 * kTileM - 1) / (2 * kTileM);
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
      kt<<<grid, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k, m.v, p, (int)n_items, nqb_max,
                                                     table);
      return cudaGetLastError();
    }
    auto kp = s.vl.cu_q != nullptr ? attn_fwd_persistent_kernel<D, BF16, true, FwdSerpentine>
                                   : attn_fwd_persistent_kernel<D, BF16, false, FwdSerpentine>;
    e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, CP::kSmemBytes);
    if (e != cudaSuccess) return e;
    kp<<<grid, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k, m.v, p, (int)n_items, nqb_max,
                                                   FwdSerpentine{});
    return cudaGetLastError();
  }
  dim3 grid(nqb_max, s.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(m.q, m.k, m.v, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const Maps& m, const Shape& s, void* o, float* lse, cudaStream_t st) {
  if (s.d > 64) return s.bf16 ? launch_fwd_t<128, true>(m, s, o, lse, st)
                                : launch_fwd_t<128, false>(m, s, o, lse, st);
  return s.bf16 ? launch_fwd_t<64, true>(m, s, o, lse, st)
                : launch_fwd_t<64, false>(m, s, o, lse, st);
}

ATTN_DEFINE_STATUS_READER(status_fwd)

}  // namespace attn
