"""The persistent kernels' item tables (csrc/schedule.h) on the CPU: the greedy builder the
launchers use, compiled into a small host program with g++.

For every shape tried, the table must list each item exactly once (an item missing from it
would leave a block of outputs unwritten; one listed twice would be computed twice), give
each CTA a contiguous run in start[], and - the reason it exists - keep the busiest CTA
close to the mean load when items differ in cost (causal attention) over few rounds.
"""
import json
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_tcgen05_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <vector>
#include "schedule.h"
using namespace attn;

// Causal forward-like costs: item x of a slice (longest first) covers 2 * (per - x) blocks,
// plus one for its fixed cost; full attention: all equal.
int main() {
  const int shapes[][4] = {  // slices, per_slice, G, causal
      {128, 16, 152, 1}, {16, 64, 152, 1}, {1024, 4, 152, 1}, {64, 16, 152, 1},
      {3, 50, 152, 1},   {7, 33, 100, 1},  {200, 8, 152, 0},  {1, 14336, 255, 1},
      {896, 16, 152, 1}, {5, 31, 17, 1}};
  std::printf("[");
  bool first = true;
  static ItemTable t;
  for (const auto& sh : shapes) {
    const int slices = sh[0], per = sh[1], G = sh[2], causal = sh[3];
    std::vector<long long> cost(per);
    for (int x = 0; x < per; ++x) cost[x] = (causal ? 2LL * (per - x) : 2LL * per) + 1;
    const int W = item_table_window(slices, 2LL << 20);
    greedy_item_table(slices, per, [&](int, int x) { return cost[x]; }, W, G, t);
    const long long n = (long long)slices * per;
    std::vector<int> seen(n, 0);
    int bad = 0;
    long long max_load = 0, total = 0;
    for (int c = 0; c < G; ++c) {
      if (t.start[c + 1] < t.start[c]) ++bad;
      long long load = 0;
      for (int i = t.start[c]; i < t.start[c + 1]; ++i) {
        const int item = t.items[i];
        if (item < 0 || item >= n) { ++bad; continue; }
        ++seen[item];
        load += cost[item % per];
      }
      total += load;
      if (load > max_load) max_load = load;
    }
    int missing = 0, twice = 0;
    for (long long i = 0; i < n; ++i) {
      if (seen[i] == 0) ++missing;
      if (seen[i] > 1) ++twice;
    }
    std::printf("%s{\"slices\": %d, \"per\": %d, \"G\": %d, \"causal\": %d, \"n\": %lld, "
                "\"start0\": %d, \"end\": %d, \"bad\": %d, \"missing\": %d, \"twice\": %d, "
                "\"balance\": %.6f}",
                first ? "" : ", ", slices, per, G, causal, n, (int)t.start[0],
                (int)t.start[G], bad, missing, twice,
                (double)total / G / (double)max_load);
    first = false;
  }
  std::printf("]\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    d = tmp_path_factory.mktemp("sched")
    src, exe = d / "harness.cpp", d / "harness"
    src.write_text(HARNESS)
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return json.loads(out)


def test_every_item_exactly_once(results):
    for r in results:
        assert r["bad"] == 0 and r["missing"] == 0 and r["twice"] == 0, r
        assert r["start0"] == 0 and r["end"] == r["n"], r


def test_busiest_cta_near_the_mean(results):
    for r in results:
        if r["n"] < 2 * r["G"]:
            continue  # fewer than two items per CTA: the longest item sets the pace
        # Longest-first greedy: the busiest CTA ends at most one item past the mean.
        assert r["balance"] >= 0.85, r
    # The shapes the benchmark runs (windows of 16 heads): as balanced as the whole sort.
    fwd = {(r["slices"], r["per"]): r["balance"] for r in results}
    assert fwd[(128, 16)] >= 0.98 and fwd[(1024, 4)] >= 0.975
