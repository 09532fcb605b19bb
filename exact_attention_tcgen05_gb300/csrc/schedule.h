// schedule.h - static schedules of the persistent kernels: a table that assigns work items
// to CTAs, built on the host and passed by value in the kernel's parameters.
//
// A persistent kernel's CTAs each walk a list of items. When items differ in cost (causal
// attention: a query block near the end of a sequence sees many more key blocks than one
// near the start) and there are only a few rounds of items per CTA, a fixed dealing order
// leaves the busiest CTA well above the mean. The table here comes from a longest-first
// greedy assignment: items are taken in windows of W slices (so that the CTAs working at
// one time share the K/V of a few heads in L2), sorted by cost within a window (longest
// first, slice order among equals), and each goes to the CTA that becomes free first.
#pragma once

#include <cstdint>

#include <algorithm>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

namespace attn {

// CTA c walks items[start[c]] .. items[start[c + 1] - 1]: 29 KiB, within the 32 KiB that
// kernel parameters may take.
constexpr int kItemTableMaxItems = 14336;
constexpr int kItemTableMaxCtas = 255;
struct ItemTable {
  uint16_t start[kItemTableMaxCtas + 1];
  uint16_t items[kItemTableMaxItems];
};

#ifdef __CUDACC__
// The k-th item of CTA c in the table; -1 past the end.
__device__ __forceinline__ int table_item(const ItemTable& t, int k, int c) {
  const int i = t.start[c] + k;
  return i < t.start[c + 1] ? t.items[i] : -1;
}
#endif

// Host: the greedy assignment of slices x per_slice items (item = slice * per_slice + x,
// cost[x] in any unit, the same for every slice) to G CTAs, in windows of W slices.
inline void greedy_item_table(int slices, int per_slice, const std::vector<long long>& cost,
                              int W, int G, ItemTable& t) {
  std::vector<int> by_cost(per_slice);
  for (int x = 0; x < per_slice; ++x) by_cost[x] = x;
  std::stable_sort(by_cost.begin(), by_cost.end(),
                   [&](int a, int b) { return cost[a] > cost[b]; });
  using Slot = std::pair<long long, int>;  // (busy until, CTA)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < G; ++c) free_at.push({0, c});
  const long long n = (long long)slices * per_slice;
  std::vector<int> owner(n), order;
  order.reserve(n);
  for (int s0 = 0; s0 < slices; s0 += W) {
    const int s1 = std::min(slices, s0 + W);
    for (int x : by_cost)
      for (int s = s0; s < s1; ++s) {
        const int item = s * per_slice + x;
        const Slot sl = free_at.top();
        free_at.pop();
        owner[item] = sl.second;
        order.push_back(item);
        free_at.push({sl.first + cost[x], sl.second});
      }
  }
  // Items grouped by CTA, each CTA's in assignment order.
  std::vector<int> pos(G + 1, 0);
  for (int item : order) ++pos[owner[item] + 1];
  for (int c = 0; c < G; ++c) pos[c + 1] += pos[c];
  for (int c = 0; c <= G; ++c) t.start[c] = (uint16_t)pos[c];
  for (int item : order) t.items[pos[owner[item]]++] = (uint16_t)item;
}

// Host: the last table a launcher built, keyed by its shape; `get` builds it on a miss
// (build(table)) and copies it into `out` under the lock, so concurrent calls never see a
// table being rebuilt.
struct ItemTableCache {
  std::mutex mu;
  ItemTable table;
  long long key[6] = {-1, -1, -1, -1, -1, -1};
  template <class Build>
  void get(const long long (&k)[6], int G, long long n_items, ItemTable& out, Build build) {
    std::lock_guard<std::mutex> lock(mu);
    if (std::memcmp(k, key, sizeof(key)) != 0) {
      build(table);
      std::memcpy(key, k, sizeof(key));
    }
    std::memcpy(out.start, table.start, sizeof(uint16_t) * (G + 1));
    std::memcpy(out.items, table.items, sizeof(uint16_t) * n_items);
  }
};

// Host: whether a table applies (dense causal inputs with more items than CTAs, within the
// table's size), and the window of slices whose K/V (or Q/dO) rows of `row_bytes` each
// take about 32 MiB, so that two windows in flight take half of the 126 MiB L2 (measured on
// GB300 against 48 MiB: B4 H32 N4096 forward 0.452 -> 0.433 ms, dK/dV -2%; B1 H16 N16384
// forward 1-3% slower).
inline bool item_table_applies(bool causal, bool packed, long long n_items, int G) {
  return causal && !packed && n_items > G && n_items <= kItemTableMaxItems &&
         G <= kItemTableMaxCtas;
}
inline int item_table_window(int slices, long long bytes_per_slice) {
  return (int)std::max(1LL, std::min<long long>(slices, (32LL << 20) / bytes_per_slice));
}

}  // namespace attn
