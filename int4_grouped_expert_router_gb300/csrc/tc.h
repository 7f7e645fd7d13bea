// Fifth-generation tensor core (tcgen05) helpers for sm_100-family GPUs: tensor-memory allocation,
// shared-memory matrix descriptors, the bf16 MMA with an f32 accumulator in tensor memory, commit
// to an mbarrier, and tensor-memory loads for the epilogue.
#pragma once

#include <stdint.h>

#include "pipe.h"

namespace coli {

// Allocate `ncols` (a power of two >= 32) tensor-memory columns for this CTA; one full warp
// executes it and the base address is written to `dst` in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Make this thread's generic-proxy shared-memory writes visible to the async proxy (the tensor
// core reads its operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte-swizzled layout: rows
// of 128 bytes (64 bf16 of K), 8-row groups 1024 bytes apart, tile base 1024-byte aligned.
// Fields: start address >> 4 [0,14), leading byte offset >> 4 [16,30) (unused for this layout, 1),
// stride byte offset >> 4 [32,46) = 1024 >> 4, descriptor version [46,48) = 1, layout [61,64) = 2.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(const void* tile) {
  const uint64_t addr = smem_u32(tile);
  return ((addr >> 4) & 0x3fffull) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B (both K-major), an f32
// accumulator and shape M x N: D format [4,6) = 1 (f32), A format [7,10) = 1 (bf16), B format
// [10,13) = 1 (bf16), N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t bf16_f32_idesc(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K step of 16; issued by a single thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 16 consecutive f32 columns of this thread's tensor-memory lane (the warp reads lanes
// 32 (warp % 4) .. + 31; taddr carries the lane in its upper half).
// The load and its wait are one asm statement: the destination registers are written
// asynchronously, so no instruction may read them before the wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

}  // namespace coli
