// pair.cuh - inline-PTX wrappers for kernels that run as clusters of two CTAs on two SMs (a
// "CTA pair") and issue tcgen05 MMAs with .cta_group::2: one MMA of M = 256 rows, each CTA
// holding 128 of them in its own tensor memory and shared memory, and half of the N columns
// of the B operand in its shared memory.
//
// Written from the public PTX ISA descriptions of these instructions. What the pair
// protocol built on them needs (the kernels state how they use it):
//  * %cluster_ctarank: the CTA's rank in its cluster (0 or 1 here). Rank 0 issues the
//    pair's MMAs and commits; both CTAs allocate and free tensor memory with
//    .cta_group::2 (one warp in each CTA, collectively).
//  * mapa.shared::cluster: the address of a shared variable in another CTA of the cluster;
//    mbarrier.arrive.release.cluster on such an address arrives on the other CTA's barrier,
//    and a wait with .acquire.cluster sees what the arriving thread wrote before it.
//  * tcgen05.commit.cta_group::2 ... .multicast::cluster: one arrival, on the barrier at
//    the same shared-memory offset in every CTA of the mask, once the MMAs the thread
//    issued before it are complete.
//  * barrier.cluster: the hardware barrier of all threads of the cluster, used once at
//    start-up (every thread of both CTAs reaches it unconditionally, before any remote
//    access); the exit handshake is a bounded mbarrier wait instead.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace attn {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster (all must reach it).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the variable at shared::cta address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// 32-bit load from another CTA's shared memory (shared::cluster address).
__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t caddr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(caddr) : "memory");
  return v;
}

// Arrive on a barrier given by its shared::cluster address (this CTA's or the peer's),
// releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr)
               : "memory");
}

// One arrival per warp on a barrier given by its shared::cluster address (see warp_arrive).
__device__ __forceinline__ void warp_arrive_cluster(uint32_t caddr) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive_cluster(caddr);
}

__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded waits with cluster-scope acquire, for barriers that receive arrivals from the
// other CTA of the pair (as mbar_wait otherwise).
__device__ __forceinline__ bool mbar_poll_cluster(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit, volatile int* abort,
                                                  int where) {
  if (mbar_test_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = clock64();
  while (true) {
    if (mbar_test_wait_cluster(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (clock64() - t0 > limit) {
      record_timeout(where);
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit, volatile int* abort,
                                                  int where) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = clock64();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (clock64() - t0 > limit) {
      record_timeout(where);
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}

// ------------------------------------------------------------------------------------
// tcgen05 with .cta_group::2
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem, 128 rows in each CTA] (+)= A[smem, 128 rows in each CTA] * B[smem, N/2 columns
// in each CTA]; descriptors name this CTA's shared memory, the peer's is read at the same
// offsets. Issued by one thread of rank 0.
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// As mma_ss_pair with A from tensor memory (each CTA's own 128 lanes at a_tmem).
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One arrival on the barrier at `bar`'s offset in each CTA of `cta_mask` once every pair
// MMA this thread issued so far is complete.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

}  // namespace attn
