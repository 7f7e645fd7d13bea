// Device helpers for streaming kernels on sm_100-family GPUs: mbarriers, bulk asynchronous copies
// (TMA) global -> shared memory, and programmatic dependent launch controls.
// Every wait is bounded: a waiting thread polls its mbarrier phase (or, with COLI_WAIT_SPIN=0,
// sleeps in mbarrier.try_wait until the phase completes) and gives up after kWaitLimitNs of
// wall-clock time; the caller then records COLI_E_TIMEOUT in the context's error word instead of
// hanging.
#pragma once

#include <stdint.h>

namespace coli {

constexpr uint32_t kSpinLimit = 1u << 24;          // polls of a non-sleeping test loop
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s
constexpr uint32_t kSuspendHintNs = 20000;           // longest single sleep inside try_wait

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy and the other threads.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test_parity(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

#ifndef COLI_WAIT_SPIN
#define COLI_WAIT_SPIN 1
#endif

// Wait until the phase with the given parity has completed; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
#if COLI_WAIT_SPIN
  // poll the non-blocking test: the thread sees the phase complete within a few hundred cycles
  // (a suspended try_wait can resume well after the phase completed)
  for (int i = 0; i < 64; i++)
    if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test_wait(bar, parity)) {
    __nanosleep(32);
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
#else
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
#endif
}

// Wait until the phase with the given parity has completed, suspended in mbarrier.try_wait (the
// thread issues nothing while the hardware holds it) instead of polling; false after limit_ns. For
// kernels with many waiting warps, whose polling would take issue slots from the warps with work.
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_test_parity(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test_parity(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from global to shared
// memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-first policy (the weights are streamed once per call).
__device__ __forceinline__ void bulk_g2s_stream(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D tiled TMA load of the box at element coordinates (x, y) of `map` (a tensor map in global,
// constant or parameter memory) into shared memory; completion on `bar` as transaction bytes.
// x times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 cache policy (from createpolicy) for the lines the copy brings in.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const void* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ int ld_volatile_int(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

// Bring a TMA descriptor (in global memory) into the copy engine's descriptor cache ahead of use.
__device__ __forceinline__ void prefetch_tensormap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// Prefetch one 128-byte line into L2 (a hint; no fault on any address of a live allocation).
__device__ __forceinline__ void prefetch_l2_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Programmatic dependent launch: wait for the preceding grid's completion and memory flush /
// allow the next grid in the stream to start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over a subset of the CTA's warps (id 1..15; count a multiple of 32).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads: every thread gets the
// same answer, so a collective decision (e.g. to stop after a timed-out wait) stays uniform.
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.cta.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p))
               : "memory");
  return v;
}

__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)) : "memory");
  return v;
}

__device__ __forceinline__ float lds32f(const void* p) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

__device__ __forceinline__ int ld_cg_i32(const int* p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Barrier over every CTA of a cooperative launch (all CTAs are resident). `count` only grows: CTA
// arrivals of this and every earlier use of the same word, G = gridDim.x per use, so this use is
// complete when the count reaches the next multiple of G above the value this CTA saw. Nothing is
// reset, and the last CTA to arrive leaves at once. Every thread's global writes before the call
// are visible to every thread after it. Returns false (the wait gave up after limit_ns)
// uniformly across the CTA. `arrive` false: this CTA waits without arriving (a test of the give-up
// path: the others then time out).
__device__ __forceinline__ bool grid_barrier(unsigned long long* count, uint64_t limit_ns = kWaitLimitNs,
                                             bool arrive = true) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned long long G = gridDim.x;
    unsigned long long old;
    if (arrive) {
      asm volatile("atom.add.release.gpu.u64 %0, [%1], 1;" : "=l"(old) : "l"(count) : "memory");
    } else {
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(old) : "l"(count) : "memory");
    }
    const unsigned long long target = (old / G + 1) * G;
    if (old + 1 != target) {
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        unsigned long long now;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(now) : "l"(count) : "memory");
        if (now >= target) break;
        if (globaltimer_ns() - t0 > limit_ns) {
          ok = 0;
          break;
        }
      }
    } else {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

}  // namespace coli
