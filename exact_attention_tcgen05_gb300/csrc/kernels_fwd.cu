// kernels_fwd.cu - instantiation and launch of the forward kernel.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
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

// Key blocks item `x` of a dense slice works through (the larger of its two tiles; the
// same geometry as fwd_item_geom).
static int fwd_item_blocks(const Shape& s, int nqb, int x) {
  const int nkb = (s.Nk + kTileN - 1) / kTileN;
  const int off = s.Nk - s.N;
  const int q0 = (nqb - 1 - x) * 2 * kTileM;
  const int ntiles = (q0 + kTileM < s.N) ? 2 : 1;
  int n = 0;
  for (int t = 0; t < ntiles; ++t)
    n = std::max(n, s.causal ? std::min(nkb, (q0 + t * kTileM + kTileM - 1 + off) / kTileN + 1)
                             : nkb);
  return n;
}

// A longest-first greedy assignment of the persistent forward's items to G CTAs, for
// dense causal inputs: the items of a window of W heads, sorted by key blocks (longest
// first, head order among equals), each go to the CTA that becomes free first, counting
// one block more per item for its fixed cost. W keeps the K/V of the heads in flight (at
// most two windows) within about 96 MiB of the 126 MiB L2. False: not worth it or too
// large for the table (then the serpentine order runs). The last table is kept (one entry
// keyed by the shape) and copied into `out` under the lock.
static bool fwd_schedule(const Shape& s, int nqb, int G, FwdSched& out) {
  const long long n_items = (long long)nqb * s.BH;
  if (!s.causal || s.vl.cu_q != nullptr || n_items <= G || n_items > kFwdSchedMaxItems ||
      G > kFwdSchedMaxCtas)
    return false;
  static std::mutex mu;
  static FwdSched table;
  static long long key[6] = {-1, -1, -1, -1, -1, -1};
  const long long k[6] = {s.BH, s.N, s.Nk, s.d, G, nqb};
  std::lock_guard<std::mutex> lock(mu);
  if (std::memcmp(k, key, sizeof(k)) != 0) {
    std::vector<int> len(nqb);
    for (int x = 0; x < nqb; ++x) len[x] = fwd_item_blocks(s, nqb, x);
    std::vector<int> by_len(nqb);  // x values, longest first (x ascending among equals)
    for (int x = 0; x < nqb; ++x) by_len[x] = x;
    std::stable_sort(by_len.begin(), by_len.end(), [&](int a, int b) { return len[a] > len[b]; });
    const long long kv_bytes = 4LL * s.Nk * s.d;  // K and V of one head, 16-bit
    const int W = (int)std::max(1LL, std::min<long long>(s.BH, (48LL << 20) / kv_bytes));
    using Slot = std::pair<long long, int>;  // (busy until, CTA)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
    for (int c = 0; c < G; ++c) free_at.push({0, c});
    std::vector<int> owner(n_items), order;
    order.reserve(n_items);
    for (int h0 = 0; h0 < s.BH; h0 += W) {
      const int h1 = std::min(s.BH, h0 + W);
      for (int x : by_len)
        for (int h = h0; h < h1; ++h) {
          const int item = h * nqb + x;
          Slot sl = free_at.top();
          free_at.pop();
          owner[item] = sl.second;
          order.push_back(item);
          free_at.push({sl.first + len[x] + 1, sl.second});
        }
    }
    // Items grouped by CTA, each CTA's in assignment order.
    std::vector<int> count(G + 1, 0);
    for (int item : order) ++count[owner[item] + 1];
    for (int c = 0; c < G; ++c) count[c + 1] += count[c];
    for (int c = 0; c <= G; ++c) table.start[c] = (uint16_t)count[c];
    for (int item : order) table.items[count[owner[item]]++] = (uint16_t)item;
    std::memcpy(key, k, sizeof(k));
  }
  std::memcpy(out.start, table.start, sizeof(uint16_t) * (G + 1));
  std::memcpy(out.items, table.items, sizeof(uint16_t) * n_items);
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
    static thread_local FwdSched table;  // 29 KiB: not on the stack
    if (fwd_schedule(s, nqb_max, grid, table)) {
      auto kt = attn_fwd_persistent_kernel<D, BF16, false, FwdSched>;
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
