// kernels_dkv.cu - instantiation and launch of the backward dK/dV kernel.
#include <algorithm>
#include <cstdlib>
#include <vector>

#include "bwd_dkv_persistent.cuh"
#include "bwd_wide.cuh"
#include "launch.h"

namespace attn {

static int sm_count_dkv() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

// Which dK/dV kernel: the persistent one (bwd_dkv_persistent.cuh) when work items are short,
// where the one-item kernel's fixed cost per CTA dominates: a key block meets fewer than 8
// query blocks on average (causal), or at most 8 (non-causal: every item is equally long,
// and B16 H32 N1024 d128 ran 0.521 -> 0.485 ms on GB300, while causal N2048 ran 1% slower);
// otherwise one CTA per key block. Dense causal inputs with more items than CTAs get a
// greedy table (schedule.h) instead of the pairs; with it the persistent kernel won or tied
// on every causal shape measured (B4 H32 N4096: 0.786 -> 0.772 ms; at d = 64 also against
// the one-item kernel's K_j, V_j in tensor memory: B8 H32 N2048 0.394 -> 0.349 ms), so it
// always runs there. ATTN_BWD_PERSISTENT = 0 / 1 forces either (both give the same bits;
// the persistent one keeps K_j, V_j in shared memory).
static bool use_persistent_dkv(const Shape& s, bool kv_tmem) {
  static const int forced = [] {
    const char* e = std::getenv("ATTN_BWD_PERSISTENT");
    return e == nullptr ? -1 : (e[0] == '0' ? 0 : 1);
  }();
  if (forced >= 0) return forced == 1;
  const long long n_items = (long long)((s.Nk + kTileN - 1) / kTileN) * s.BH;
  if (item_table_applies(s.causal, s.vl.cu_q != nullptr, s.host_cu_q != nullptr, n_items,
                         (int)std::min<long long>(n_items, sm_count_dkv())))
    return true;
  if (kv_tmem) return false;
  const int nb = (s.N + kTileM - 1) / kTileM;
  return s.causal ? (nb + 1) / 2 < 8 : nb <= 8;
}

// The persistent dK/dV's table (schedule.h) for causal dense inputs, or packed batches
// whose host lengths are known, with more items than CTAs: item slot jb of a slice is key
// block jb, its cost the query blocks that see it + 1 (the geometry of dkv_item_geom; a
// key block of a sequence without queries costs 1: its gradients are zero-filled), windows
// of heads by their Q/dO bytes. False: the long/short pairs run.
static bool dkv_schedule(const Shape& s, int nkb_max, int G, ItemTable& out) {
  const bool packed = s.vl.cu_q != nullptr;
  const long long n_items = (long long)nkb_max * s.BH;
  if (!item_table_applies(s.causal, packed, s.host_cu_q != nullptr, n_items, G)) return false;
  static ItemTableCache cache;
  const long long k[8] = {s.BH, s.N, s.Nk, s.d, G, nkb_max, s.causal ? 1 : 0,
                          lengths_hash(s.host_cu_q, s.host_cu_k, s.vl_b)};
  cache.get(k, G, n_items, out, [&](ItemTable& t) {
    const long long qdo_bytes =
        packed ? 4LL * std::max(1, s.vl.total_q / std::max(1, s.vl_b)) * s.d : 4LL * s.N * s.d;
    auto cost = [&](int bh, int jb) -> long long {
      int nq, nk;
      slice_lengths(s, bh, nq, nk);
      const int j0 = jb * kTileN;
      if (j0 >= nk) return 0;
      const int nb = (nq + kTileM - 1) / kTileM, off = nk - nq;
      const int i_first = (s.causal && j0 > off) ? (j0 - off) / kTileM : 0;
      return (nq == 0 ? 0 : std::max(0, nb - i_first)) + 1;
    };
    greedy_item_table(s.BH, nkb_max, cost, item_table_window(s.BH, qdo_bytes), G, t);
  });
  return true;
}

template <int D, bool BF16>
static cudaError_t launch_dkv_t(const Maps& m, const Shape& s, const void* q, const void* k,
                                const void* v, const void* d_o, const float* lse,
                                const float* delta, void* dk, void* dv, cudaStream_t st) {
  using C = DkvCfg<D>;
  // d = 64: K_j, V_j in tensor memory when a key block meets about eight or more query
  // blocks (the one-time row copy costs more than it saves on shorter work).
  const bool kv_tmem = D == 64 && (s.causal ? s.N >= 2048 : s.N >= 1024);
  auto kern = s.vl.cu_q != nullptr
                  ? (kv_tmem ? attn_bwd_dkv_kernel<D, BF16, true, D == 64>
                             : attn_bwd_dkv_kernel<D, BF16, true, false>)
                  : (kv_tmem ? attn_bwd_dkv_kernel<D, BF16, false, D == 64>
                             : attn_bwd_dkv_kernel<D, BF16, false, false>);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  BwdParams p;
  p.in_q = q;
  p.in_k = k;
  p.in_v = v;
  p.in_do = d_o;
  p.lse = lse;
  p.delta = delta;
  p.out0 = dk;
  p.out1 = dv;
  p.dh = s.d;
  p.N = s.N;
  p.Nk = s.Nk;
  p.vl = s.vl;
  p.causal = s.causal ? 1 : 0;
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.wait_limit = s.wait_limit;
  p.stall = s.stall;
  const int nkb_max = (s.Nk + kTileN - 1) / kTileN;  // packed batches: the longest sequence
  if (use_persistent_dkv(s, kv_tmem)) {
    using CP = DkvPCfg<D>;
    const int npairs = (nkb_max + 1) / 2;
    const long long n_pairs = (long long)npairs * s.BH;
    const int gt = (int)std::min<long long>((long long)nkb_max * s.BH, sm_count_dkv());
    static thread_local ItemTable table;  // 29 KiB: not on the stack
    if (dkv_schedule(s, nkb_max, gt, table)) {
      auto kt = s.vl.cu_q != nullptr ? attn_bwd_dkv_persistent_kernel<D, BF16, true, ItemTable>
                                     : attn_bwd_dkv_persistent_kernel<D, BF16, false, ItemTable>;
      e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, CP::kSmemBytes);
      if (e != cudaSuccess) return e;
      kt<<<gt, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k, m.v, m.d_o, m.dk, m.dv, p,
                                                   (int)n_pairs, npairs, nkb_max, table);
      return cudaGetLastError();
    }
    auto kp = s.vl.cu_q != nullptr
                  ? attn_bwd_dkv_persistent_kernel<D, BF16, true, PairSchedule>
                  : attn_bwd_dkv_persistent_kernel<D, BF16, false, PairSchedule>;
    e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, CP::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<long long>(n_pairs, sm_count_dkv());
    kp<<<grid, CP::kThreads, CP::kSmemBytes, st>>>(m.q, m.k, m.v, m.d_o, m.dk, m.dv, p,
                                                   (int)n_pairs, npairs, nkb_max, PairSchedule{});
    return cudaGetLastError();
  }
  // One CTA per 128-key block.
  dim3 grid(nkb_max, s.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(m.q, m.k, m.v, m.d_o, p);
  return cudaGetLastError();
}

cudaError_t launch_dkv(const Maps& m, const Shape& s, const void* q, const void* k,
                       const void* v, const void* d_o, const float* lse, const float* delta,
                       void* dk, void* dv, cudaStream_t st) {
  if (s.d > 128) {
    // two passes (dK and dV together would need 512 accumulator columns): dV with K_j
    // resident, then dK with K_j, V_j resident; Q_i, dO_i streamed in both
    cudaError_t e = s.bf16 ? launch_bwd_wide<kWideDV, true>(m.k, m.q64, m.do64, k, s, lse,
                                                            delta, dk, dv, st)
                           : launch_bwd_wide<kWideDV, false>(m.k, m.q64, m.do64, k, s, lse,
                                                             delta, dk, dv, st);
    if (e != cudaSuccess) return e;
    return s.bf16 ? launch_bwd_wide<kWideDK, true>(m.k, m.q64, m.do64, v, s, lse, delta, dk, dv,
                                                   st)
                  : launch_bwd_wide<kWideDK, false>(m.k, m.q64, m.do64, v, s, lse, delta, dk,
                                                    dv, st);
  }
  if (s.d > 64)
    return s.bf16 ? launch_dkv_t<128, true>(m, s, q, k, v, d_o, lse, delta, dk, dv, st)
                  : launch_dkv_t<128, false>(m, s, q, k, v, d_o, lse, delta, dk, dv, st);
  return s.bf16 ? launch_dkv_t<64, true>(m, s, q, k, v, d_o, lse, delta, dk, dv, st)
                : launch_dkv_t<64, false>(m, s, q, k, v, d_o, lse, delta, dk, dv, st);
}

ATTN_DEFINE_STATUS_READER(status_dkv)

}  // namespace attn
