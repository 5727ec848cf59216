// Inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM alloc, MMA, commit, load) and a bounded wait.
//
// Every wait on an mbarrier in this library goes through wait_bounded: it
// polls with try_wait and gives up after kWaitLimitNs of %globaltimer time,
// setting the CTA's abort flag and the device status word, so that a broken
// pipeline returns an error instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lmoe {

constexpr unsigned kStatusTimeout = 1u;    // LATENTMOE_STATUS_TIMEOUT
constexpr unsigned kStatusBadExpert = 2u;  // LATENTMOE_STATUS_BAD_EXPERT
constexpr unsigned kStatusRounds = 4u;     // LATENTMOE_STATUS_ROUNDS
constexpr unsigned kStatusBounds = 8u;     // LATENTMOE_STATUS_BOUNDS (bounds-checked build)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legal wait
// Suspend-time hint of every try_wait: a waiting thread may sleep up to this
// long (it wakes as soon as the phase completes) instead of returning to the
// poll loop, so idle roles issue fewer instructions (less power under the
// power cap).
constexpr uint32_t kWaitHintNs = 20000;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounds-checked debug build (compiled with -DLMOE_BOUNDS): every epilogue
// store, scatter write and combine read asks in_bounds(i, n, status) whether
// row i of a buffer of n rows exists; an access outside is skipped and sets
// kStatusBounds in the device status word (nothing traps). In the regular
// build in_bounds is the constant true and compiles away.
#ifdef LMOE_BOUNDS
__device__ __forceinline__ bool in_bounds(long long i, long long n, unsigned* status) {
  if (i >= 0 && i < n) return true;
  if (status != nullptr) atomicOr(status, kStatusBounds);
  return false;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(long long, long long, unsigned*) {
  return true;
}
#endif

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kWaitHintNs)
      : "memory");
  return done != 0;
}

// Wait until the phase with the given parity has completed. Returns false if
// the CTA's abort flag was raised or the time limit passed (then it raises the
// abort flag itself and ORs kStatusTimeout into *status).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, unsigned* status,
                                             uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// All lanes of a warp wait together: lane 0 polls, the verdict is broadcast,
// then the other lanes observe the completed phase themselves.
__device__ __forceinline__ bool warp_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, unsigned* status) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) ok = wait_bounded(bar, parity, abort_flag, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok && lane != 0) ok = mbar_try_wait(bar, parity) ? 1 : wait_bounded(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Teardown variant: no abort check (used to drain copies already in flight).
__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// ---------------------------------------------------------------- programmatic dependent launch
// The forward's kernels are enqueued with programmatic stream serialization,
// so a kernel's CTAs may be scheduled (and run their own shared-memory and
// TMEM set-up) while the kernel before it is still finishing. Every kernel
// therefore calls pdl_wait() before its first read of anything an earlier
// kernel wrote: it returns once the preceding kernel has completed and its
// writes are visible (at once for a kernel launched without the attribute).
// Since every kernel waits before it completes, completion is transitive down
// the chain. pdl_launch_dependents() then lets the next kernel be scheduled;
// it is called after the wait, so at most one kernel runs ahead.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at (c0 = inner element index, c1 = row) into
// shared memory, completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// 3-D tiled load of the box at (c0, c1, c2) (c0 innermost).
__device__ __forceinline__ void tma_load_3d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// A 16-byte global store with an L2 eviction-priority policy.
__device__ __forceinline__ void st_global_u4_hint(uint4* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// ---------------------------------------------------------------- cross-CTA completion counts
// A 32-bit load with acquire semantics at GPU scope: writes released before
// the value was stored (by any CTA) are visible after it.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Orders this thread's earlier global accesses (here: the acquire above)
// before its later async-proxy accesses (TMA loads of what other CTAs wrote).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with kind::f8f6f4 (both operands E4M3 per the instruction
// descriptor, 32 elements = 32 bytes of K per instruction, fp32 accumulate).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all tcgen05 ops issued so far by this thread finish.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (lane base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_8cols(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

// Named barrier for `count` threads (a multiple of 32) with id 1..15.
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 128 bytes (64 elements), 8-row groups 1024 bytes
// apart. Bits: [0,14) start >> 4, [16,30) leading offset >> 4 (unused for
// swizzled K-major, set to 1), [32,46) stride offset >> 4 = 1024 >> 4,
// [46,48) version 1, [61,64) layout 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* tile) {
  const uint64_t addr = smem_addr(tile);
  return ((addr & 0x3FFFFull) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}

// Same for a K-major bf16 tile written by TMA with 64-byte swizzle: rows of
// 64 bytes (32 elements), 8-row groups 512 bytes apart; layout type 4.
__device__ __forceinline__ uint64_t smem_desc_sw64(const void* tile) {
  const uint64_t addr = smem_addr(tile);
  return ((addr & 0x3FFFFull) >> 4) | (1ull << 16) | (32ull << 32) | (1ull << 46) |
         (4ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits [4,6) = 1),
// A and B bf16 (bits [7,10) and [10,13) = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits [17,23), M >> 4 in bits [24,29).
__host__ __device__ constexpr uint32_t instr_desc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with A and B both E4M3 (format code 0
// in bits [7,10) and [10,13)), fp32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t instr_desc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// SiLU(a) = a * sigmoid(a) with sigmoid(a) = (1 + tanh(a/2)) / 2, i.e.
// a/2 + (a/2) tanh(a/2): one special-function op (the hardware tanh, whose
// error is about 2^-11 of the result) and two FP32 ops, against two
// special-function ops for a / (1 + e^-a). The grouped epilogues evaluate it
// for every element of h and are bound by the special-function pipe; the
// error stays below the bf16 rounding of h (2^-9).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// SiLU(a) = h + h tanh(h) with h = a / 2, from h. Callers that scale the
// accumulator anyway pass the scale times 1/2 (exact: a power of two) and
// save the halving.
__device__ __forceinline__ float silu_from_half(float h) { return fmaf(h, tanh_approx(h), h); }
__device__ __forceinline__ float silu(float a) { return silu_from_half(0.5f * a); }

}  // namespace lmoe
