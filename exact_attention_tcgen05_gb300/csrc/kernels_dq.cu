// kernels_dq.cu - instantiation and launch of the backward dQ kernel.
#include <algorithm>
#include <cstdlib>
#include <vector>

#include "bwd_dq_persistent.cuh"
#include "bwd_wide.cuh"
#include "launch.h"

namespace attn {

static int sm_count_dq() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

// Which dQ kernel: the persistent one (bwd_dq_persistent.cuh) or one CTA per item. The
// one-item kernel pays a fixed cost per CTA (about 7 us on GB300, as much as 8 blocks of
// work) but the hardware schedules its CTAs dynamically; the persistent kernel removes most
// of that cost, but its static long/short pairs end when the busiest SM ends: after
// ceil(pairs / SMs) rounds, against pairs / SMs rounds of work. Measured on GB300: the
// persistent kernel wins for items shorter than 8 key blocks whatever the rounds, wins or
// ties up to 16 blocks when the last round is at least 95% full (B4 H32 N4096 causal:
// 13.5 rounds, 0.621 -> 0.599 ms), and ties or loses for longer items or emptier last
// rounds (10.1 rounds at N3072 and N6144; B2 H32 N8192 d64 full: 1.375 -> 1.430 ms).
// Dense causal inputs with more items than CTAs get a greedy table (schedule.h) instead of
// the pairs, which balances any number of rounds; with it the persistent kernel won or tied
// on every causal shape measured (N = 1024-16384, d = 64 and 128; B4 H32 N4096:
// 0.602 -> 0.577 ms), so it always runs there.
// ATTN_BWD_PERSISTENT = 0 / 1 forces either (both give the same bits).
static bool use_persistent_dq(const Shape& s) {
  static const int forced = [] {
    const char* e = std::getenv("ATTN_BWD_PERSISTENT");
    return e == nullptr ? -1 : (e[0] == '0' ? 0 : 1);
  }();
  if (forced >= 0) return forced == 1;
  const long long n_items = (long long)((s.N + kTileM - 1) / kTileM) * s.BH;
  if (item_table_applies(s.causal, s.vl.cu_q != nullptr, s.host_cu_q != nullptr, n_items,
                         (int)std::min<long long>(n_items, sm_count_dq())))
    return true;
  const int nkb = (s.Nk + kTileN - 1) / kTileN;
  const int blocks_per_item = s.causal ? (nkb + 1) / 2 : nkb;
  if (blocks_per_item < 8) return true;
  // Packed batches: pairs of sequences shorter than the longest are skipped, so the round
  // count says little about the balance (an 8-sequence batch of 601-4008 tokens took
  // 1.54 -> 1.57 ms per step with the persistent dQ).
  if (blocks_per_item > 16 || s.vl.cu_q != nullptr) return false;
  const long long n_pairs = (long long)(((s.N + kTileM - 1) / kTileM + 1) / 2) * s.BH;
  const long long sms = sm_count_dq();
  const long long rounds = (n_pairs + sms - 1) / sms;
  return n_pairs * 20 >= rounds * sms * 19;
}

// The persistent dQ's table (schedule.h) for causal dense inputs, or packed batches whose
// host lengths are known, with more items than CTAs: item slot x of a slice is query block
// nb - 1 - x (causal) or x, its cost the key blocks it sees + 1 (the geometry of
// dq_item_geom), windows of heads by their K/V bytes. False: the long/short pairs run.
static bool dq_schedule(const Shape& s, int nb_max, int G, ItemTable& out) {
  const bool packed = s.vl.cu_q != nullptr;
  const long long n_items = (long long)nb_max * s.BH;
  if (!item_table_applies(s.causal, packed, s.host_cu_q != nullptr, n_items, G)) return false;
  static ItemTableCache cache;
  const long long k[8] = {s.BH, s.N, s.Nk, s.d, G, nb_max, s.causal ? 1 : 0,
                          lengths_hash(s.host_cu_q, s.host_cu_k, s.vl_b)};
  cache.get(k, G, n_items, out, [&](ItemTable& t) {
    const long long kv_bytes =
        packed ? 4LL * std::max(1, s.vl.total_k / std::max(1, s.vl_b)) * s.d : 4LL * s.Nk * s.d;
    auto cost = [&](int bh, int x) -> long long {
      int nq, nk;
      slice_lengths(s, bh, nq, nk);
      const int nb = (nq + kTileM - 1) / kTileM;
      if (x >= nb) return 0;
      const int nkb = (nk + kTileN - 1) / kTileN;
      const int i0 = (s.causal ? nb - 1 - x : x) * kTileM;
      const int n = s.causal ? std::min(nkb, (i0 + kTileM - 1 + nk - nq) / kTileN + 1) : nkb;
      return n + 1;
    };
    greedy_item_table(s.BH, nb_max, cost, item_table_window(s.BH, kv_bytes), G, t);
  });
  return true;
}

template <int D, bool BF16>
static cudaError_t launch_dq_t(const Maps& m, const Shape& s, const void* q,
                               const void* d_o, const float* lse,
                               const float* delta, void* dq, cudaStream_t st) {
  using C = DqCfg<D>;
  auto kern = s.vl.cu_q != nullptr ? attn_bwd_dq_kernel<D, BF16, true>
                                   : attn_bwd_dq_kernel<D, BF16, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  BwdParams p;
  p.in_q = q;
  p.in_k = nullptr;
  p.in_v = nullptr;
  p.in_do = d_o;
  p.lse = lse;
  p.delta = delta;
  p.out0 = dq;
  p.out1 = nullptr;
  p.dh = s.d;
  p.N = s.N;
  p.Nk = s.Nk;
  p.vl = s.vl;
  p.causal = s.causal ? 1 : 0;
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  p.stall = s.stall;
  const int nb_max = (s.N + kTileM - 1) / kTileM;  // packed batches: the longest sequence
  if (use_persistent_dq(s)) {
    using CP = DqPCfg<D>;
    const int npairs = (nb_max + 1) / 2;
    const long long n_pairs = (long long)npairs * s.BH;
    const int gt = (int)std::min<long long>((long long)nb_max * s.BH, sm_count_dq());
    static thread_local ItemTable table;  // 29 KiB: not on the stack
    if (dq_schedule(s, nb_max, gt, table)) {
      auto kt = s.vl.cu_q != nullptr ? attn_bwd_dq_persistent_kernel<D, BF16, true, ItemTable>
                                     : attn_bwd_dq_persistent_kernel<D, BF16, false, ItemTable>;
      e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, CP::kSmemBytes);
      if (e != cudaSuccess) return e;
      kt<<<gt, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k, m.v, m.d_o, m.dq, p, (int)n_pairs,
                                                   npairs, nb_max, table);
      return cudaGetLastError();
    }
    auto kp = s.vl.cu_q != nullptr ? attn_bwd_dq_persistent_kernel<D, BF16, true, PairSchedule>
                                   : attn_bwd_dq_persistent_kernel<D, BF16, false, PairSchedule>;
    e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, CP::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<long long>(n_pairs, sm_count_dq());
    kp<<<grid, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k, m.v, m.d_o, m.dq, p, (int)n_pairs,
                                                   npairs, nb_max, PairSchedule{});
    return cudaGetLastError();
  }
  // One CTA per 128-row query block.
  dim3 grid(nb_max, s.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(m.q, m.k, m.v, m.d_o, p);
  return cudaGetLastError();
}

cudaError_t launch_dq(const Maps& m, const Shape& s, const void* q, const void* d_o,
                       const float* lse, const float* delta,
                      void* dq, cudaStream_t st) {
  if (s.d > 128)  // Q_i, dO_i resident; K_j, V_j streamed
    return s.bf16 ? launch_bwd_wide<kWideDQ, true>(m.q, m.k64, m.v64, d_o, s, lse, delta, dq,
                                                   nullptr, st)
                  : launch_bwd_wide<kWideDQ, false>(m.q, m.k64, m.v64, d_o, s, lse, delta, dq,
                                                    nullptr, st);
  if (s.d > 64) return s.bf16 ? launch_dq_t<128, true>(m, s, q, d_o, lse, delta, dq, st)
                                : launch_dq_t<128, false>(m, s, q, d_o, lse, delta, dq, st);
  return s.bf16 ? launch_dq_t<64, true>(m, s, q, d_o, lse, delta, dq, st)
                : launch_dq_t<64, false>(m, s, q, d_o, lse, delta, dq, st);
}

ATTN_DEFINE_STATUS_READER(status_dq)

}  // namespace attn
