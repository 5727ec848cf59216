// Inline-PTX wrappers for CTA pairs (a cluster of 2 CTAs on two SMs that run
// tcgen05 MMAs with cta_group::2: M = 256 split over the pair's tensor
// memories, the B operand split by rows between the pair's shared memories).
//
// Rules this library follows for a pair kernel:
// - Every tcgen05 instruction of the kernel uses cta_group::2.
// - TMEM is allocated, relinquished and freed by one warp in each CTA of the
//   pair together; both CTAs get the same columns.
// - Only the even CTA (rank 0, the leader) issues MMAs and commits; commits
//   arrive on the barrier at the same offset in both CTAs (multicast).
// - TMA loads of either CTA land in the issuing CTA's shared memory and
//   complete their bytes on the leader's barrier, whose expected byte count
//   the leader sets for both CTAs.
// - Barriers are initialised and the pair synchronises (barrier.cluster)
//   before any CTA touches the other's barriers, and again before TMEM is
//   freed and the CTAs exit.
// Every wait stays bounded as in ptx.cuh; a CTA that gives up also raises the
// other CTA's abort flag.
#pragma once

#include "ptx.cuh"

namespace lmoe {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t cta_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(cta_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kWaitHintNs)
      : "memory");
  return done != 0;
}

// Store a 32-bit value at a cluster shared-memory address (this CTA's or
// the peer's); a later release arrive orders it for the reader.
__device__ __forceinline__ void st_cluster_s32(uint32_t cluster_addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Arrive once on a barrier given by its cluster address (this CTA's or the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// wait_bounded for a pair: on timeout, also raise the peer's abort flag
// (peer_abort = cluster address of the peer CTA's flag).
__device__ __forceinline__ bool wait_bounded_pair(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, uint32_t peer_abort,
                                                  unsigned* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((++n & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1u) : "memory");
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool warp_wait_bounded_pair(uint64_t* bar, uint32_t parity,
                                                       volatile int* abort_flag,
                                                       uint32_t peer_abort, unsigned* status) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) ok = wait_bounded_pair(bar, parity, abort_flag, peer_abort, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok && lane != 0)
    ok = mbar_try_wait_cluster(bar, parity)
             ? 1
             : wait_bounded_pair(bar, parity, abort_flag, peer_abort, status);
  return __all_sync(0xffffffffu, ok) != 0;
}

// TMA loads into this CTA's shared memory that complete on the barrier at
// cluster address `bar` (the leader's).
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap* map, uint32_t bar, void* dst,
                                                 int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(const CUtensorMap* map, uint32_t bar, void* dst,
                                                 int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
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

// D (M = 256 over the pair) (+)= A B^T, bf16 operands (kind::f16).
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with E4M3 operands (kind::f8f6f4).
__device__ __forceinline__ void tc_mma_pair_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` (same offset) in every CTA of `cta_mask` when all
// tcgen05 ops issued so far by this thread finish.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(cta_mask)
      : "memory");
}

}  // namespace lmoe
