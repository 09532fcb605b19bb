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

// Host: the greedy assignment of slices x per_slice items (item = slice * per_slice + x)
// to G CTAs, in windows of W slices; cost(slice, x) in any unit, 0 for an empty slot (a
// block past its sequence's end). Within a window the items go longest first (then by x,
// then by slice); each to the CTA that becomes free first. Empty slots are still listed -
// the kernels skip them after looking at their geometry - but dealt round-robin at the
// ends of the CTAs' lists, so that no CTA collects them all.
template <class Cost>
inline void greedy_item_table(int slices, int per_slice, Cost cost, int W, int G,
                              ItemTable& t) {
  using Slot = std::pair<long long, int>;  // (busy until, CTA)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < G; ++c) free_at.push({0, c});
  const long long n = (long long)slices * per_slice;
  std::vector<int> owner(n), order, empty;
  order.reserve(n);
  struct Item {
    long long cost;
    int x, slice;
  };
  std::vector<Item> win;
  for (int s0 = 0; s0 < slices; s0 += W) {
    const int s1 = std::min(slices, s0 + W);
    win.clear();
    for (int s = s0; s < s1; ++s)
      for (int x = 0; x < per_slice; ++x) {
        const long long c = cost(s, x);
        if (c > 0)
          win.push_back({c, x, s});
        else
          empty.push_back(s * per_slice + x);
      }
    std::stable_sort(win.begin(), win.end(), [](const Item& a, const Item& b) {
      if (a.cost != b.cost) return a.cost > b.cost;
      if (a.x != b.x) return a.x < b.x;
      return a.slice < b.slice;
    });
    for (const Item& it : win) {
      const int item = it.slice * per_slice + it.x;
      const Slot sl = free_at.top();
      free_at.pop();
      owner[item] = sl.second;
      order.push_back(item);
      free_at.push({sl.first + it.cost, sl.second});
    }
  }
  for (size_t i = 0; i < empty.size(); ++i) {
    owner[empty[i]] = (int)(i % G);
    order.push_back(empty[i]);
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
  long long key[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
  template <class Build>
  void get(const long long (&k)[8], int G, long long n_items, ItemTable& out, Build build) {
    std::lock_guard<std::mutex> lock(mu);
    if (std::memcmp(k, key, sizeof(key)) != 0) {
      build(table);
      std::memcpy(key, k, sizeof(key));
    }
    std::memcpy(out.start, table.start, sizeof(uint16_t) * (G + 1));
    std::memcpy(out.items, table.items, sizeof(uint16_t) * n_items);
  }
};

// Host: a hash of a packed batch's host lengths for the cache key (0 for dense inputs). A
// collision only reuses another order of the same item slots.
inline long long lengths_hash(const int* cu_q, const int* cu_k, int n) {
  if (cu_q == nullptr) return 0;
  unsigned long long h = 1469598103934665603ull;
  for (int i = 0; i <= n; ++i) {
    h = (h ^ (unsigned)cu_q[i]) * 1099511628211ull;
    h = (h ^ (unsigned)cu_k[i]) * 1099511628211ull;
  }
  return (long long)(h >> 1);
}

// Host: whether a table applies - items of unequal cost (causal inputs, or packed
// sequences whose lengths the host knows), more items than CTAs, within the table's size -
// and the window of slices whose K/V (or Q/dO) rows take about 32 MiB, so that two windows
// in flight take half of the 126 MiB L2 (measured on GB300 against 48 MiB: B4 H32 N4096
// forward 0.452 -> 0.433 ms, dK/dV -2%; B1 H16 N16384 forward 1-3% slower).
inline bool item_table_applies(bool causal, bool packed, bool packed_lengths_known,
                               long long n_items, int G) {
  if (packed ? !packed_lengths_known : !causal) return false;
  return n_items > G && n_items <= kItemTableMaxItems && G <= kItemTableMaxCtas;
}
inline int item_table_window(int slices, long long bytes_per_slice) {
  return (int)std::max(1LL, std::min<long long>(slices, (32LL << 20) / bytes_per_slice));
}

}  // namespace attn
