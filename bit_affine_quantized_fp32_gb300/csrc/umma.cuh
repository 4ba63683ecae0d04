// umma.cuh -- 5th-generation tensor core (tcgen05) helpers for sm_103a:
// tensor-memory allocation, shared-memory matrix descriptors, the 16-bit MMA
// (A from tensor memory, B from shared memory) with fp32 accumulation in
// tensor memory, its completion barrier, and the tensor-memory stores and
// loads around it.  Inline PTX only.
//
// Operand tiles live in shared memory in the K-major layout with the 128-byte
// swizzle: a tile of 64 16-bit columns stores row r as 128 contiguous bytes
// at 128 r, its 16-byte piece c (columns 8c .. 8c + 7) at slot c ^ (r & 7);
// eight rows make a 1024-byte swizzle atom, atoms 1024 bytes apart (the
// stride byte offset).  The tile base is 1024-byte aligned, since the
// swizzle acts on the address bits themselves; the K slice kk (16 columns)
// of an MMA starts 32 kk bytes after the tile base.  Eight 16-byte stores
// to the eight pieces of one row, or to pieces whose (c ^ (r & 7)) differ,
// fall in eight distinct bank groups (one shared-memory wavefront).
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace moe {

constexpr int kUmmaRowBytes = 128;    // 64 16-bit columns
constexpr int kUmmaAtomBytes = 1024;  // 8 rows

// Byte offset of 16-bit element (r, k) (k < 64) of a K-major 128-byte-swizzled
// tile.
__host__ __device__ inline int umma_off_sw128(int r, int k) {
  return r * kUmmaRowBytes + ((((k >> 3) ^ (r & 7)) & 7) << 4) + (k & 7) * 2;
}

// Shared-memory matrix descriptor of a K-major 128-byte-swizzled tile (or of
// its K slice at saddr = base + 32 kk): start address, leading byte offset
// 16 (unused by this layout), stride byte offset 1024, descriptor version 1,
// base offset 0, layout type 2 (128-byte swizzle) in bits 61..63.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(16 >> 4) << 16;
  d |= uint64_t(kUmmaAtomBytes >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16 with fp16 A and B (both K-major, the
// A and B format fields 0) and an fp32 accumulator, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4)                       // D format: f32
         | (uint32_t(N >> 3) << 17)      // N / 8
         | (uint32_t(M >> 4) << 24);     // M / 16
}

// D[tmem] (+)= A[tmem] * B^T over K = 16: A from tensor memory (lane m =
// row m, column c = K elements 2c (low half) and 2c + 1), B from shared
// memory, issued by one thread.
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                                uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1 : 0)
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

// One 16-lane x 8-column block of tensor memory from registers (shape
// 16x256b, one repeat): thread l of the warp writes lanes L + l / 4 (r0, r1)
// and L + 8 + l / 4 (r2, r3), columns C + 2 (l % 4) (r0, r2) and
// C + 2 (l % 4) + 1 (r1, r3), where taddr = (L << 16) | C and the lanes
// L .. L + 15 lie in this warp's quarter (32 (warp % 4) ..).  Asynchronous:
// tmem_wait_st orders it before later reads by other threads.
__device__ __forceinline__ void tmem_st_16x256b(uint32_t taddr, uint32_t r0, uint32_t r1,
                                                uint32_t r2, uint32_t r3) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(taddr),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane: warp w of
// a warpgroup reads lanes 32 (w % 4) .. + 31, thread l lane 32 (w % 4) + l;
// taddr carries the lane base in bits 16..31 and the column in bits 0..15.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace moe
