// umma.cuh -- 5th-generation tensor core (tcgen05) helpers for sm_103a:
// tensor-memory allocation, shared-memory matrix descriptors, the bf16 MMA
// with fp32 accumulation in tensor memory, its completion barrier and the
// tensor-memory loads of the epilogue.  Inline PTX only.
//
// Operand tiles live in shared memory in the K-major layout without swizzle:
// 8-row x 16-byte core matrices (8 rows x 8 bf16 along K), one core matrix
// = 128 contiguous bytes, row r of it at byte 16 r.  A tile of R rows and
// KT columns stores core matrix (row block i, k block j) at
//   i * sbo + j * lbo        with lbo = 128 and sbo = (KT / 8) * 128,
// i.e. the K blocks of one 8-row block are contiguous.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace moe {

// Byte offset of element (r, k) of a K-major no-swizzle tile with KT columns.
__host__ __device__ inline int umma_off(int r, int k, int KT) {
  return (r >> 3) * (KT / 8) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

// Shared-memory matrix descriptor: start address, leading (K) and stride
// (M/N) byte offsets, descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo & 0x3FFFFu) >> 4) << 16;
  d |= uint64_t((sbo & 0x3FFFFu) >> 4) << 32;
  d |= uint64_t(1) << 46;  // version
  return d;                // base offset 0, relative LBO mode, no swizzle
}

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major) and an
// fp32 accumulator, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4)                       // D format: f32
         | (1u << 7)                     // A format: bf16
         | (1u << 10)                    // B format: bf16
         | (uint32_t(N >> 3) << 17)      // N / 8
         | (uint32_t(M >> 4) << 24);     // M / 16
}

// D[tmem] (+)= A * B^T over K = 16, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

// Arrive once on the mbarrier when every MMA issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Tensor-memory allocation by one whole warp: ncols (a power of two >= 32)
// columns; the address is written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// 8 consecutive fp32 columns of this thread's tensor-memory lane: warp w of a
// warpgroup reads lanes 32 (w % 4) .. + 31, thread l lane 32 (w % 4) + l.
// taddr carries the lane base in bits 16..31 and the column in bits 0..15.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace moe
