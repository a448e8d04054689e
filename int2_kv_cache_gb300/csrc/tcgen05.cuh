// Fifth-generation tensor cores (sm_100 family): tensor-memory allocation,
// shared-memory matrix descriptors, tcgen05.mma issue and completion, and the
// tensor-memory -> register loads of the epilogue.  Inline PTX only.
#pragma once
#include <stdint.h>

#include "async_copy.cuh"

namespace kvq {

// Tensor memory: 128 lanes x 512 columns of 32-bit cells per SM.  One warp
// allocates a power-of-two number (>= 32) of columns and frees them again; the
// base address (lane 0, first column) is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Ordering of tensor-core operations around thread synchronisation.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile stored as rows of
// 128 bytes (64 bf16) with the 128-byte swizzle (16-byte chunk c of row r at
// chunk c ^ (r % 8)), 8-row groups 1,024 bytes apart, tile base 1,024-byte
// aligned.  Fields: start address >> 4 (bits 0-13), leading-dimension offset
// >> 4 (16-29, unused for this layout), stride-dimension offset >> 4 (32-45),
// descriptor version 1 (46-47), base offset 0 (49-51), swizzle mode 2 =
// 128-byte (61-63).  Stepping K by 16 elements advances the start by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(const void* tile) {
  const uint32_t a = smem_u32(tile);
  return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major), fp32
// D, an M x N tile: D format (bits 4-5) = 1 (f32), A format (7-9) = 1 (bf16),
// B format (10-12) = 1 (bf16), N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// The mbarrier receives one arrival once every tensor-core operation issued so
// far by this thread has completed (its shared-memory operands may be reused).
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// 8 consecutive 32-bit columns of the lane this thread maps to (warp w of a
// warpgroup reads lanes 32 (w % 4) .. 32 (w % 4) + 31).  The load and its wait
// sit in one asm statement, so no use of the registers can precede the wait.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace kvq
