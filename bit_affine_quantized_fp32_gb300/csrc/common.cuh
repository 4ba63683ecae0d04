// common.cuh -- device helpers shared by the MoE kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

namespace moe {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// Workspace layout.  Every region is 256-byte aligned; the layout depends only
// on the call's shape, so any workspace of moe_workspace_bytes(max_tokens, ...)
// bytes serves every call with n_tokens <= max_tokens.
struct WsLayout {
  size_t ctrl;        // int32 control words ([0] device status), 16 KiB
  size_t logits;      // f32 [T][E]
  size_t gate_logit;  // f32 [T]
  size_t xperm;       // u16 [T][H]   activations, k-permuted inside 8-blocks
  size_t xsum;        // f32 [T][H/64] per-64-group sums of x
  size_t idx;         // i32 [T][k]
  size_t w;           // f32 [T][k]
  size_t sgw;         // f32 [T]
  size_t offsets;     // i32 [E+1]
  size_t perm;        // i32 [T*k]
  size_t nss;         // i32 [1]   number of sub-slots
  size_t ss_e;        // i32 [maxss] expert of each sub-slot
  size_t ss_off;      // i32 [maxss] first bucket position
  size_t ss_cnt;      // i32 [maxss] tokens (1..8)
  size_t ss_rows;     // i32 [maxss][8] token of each sub-slot position
  size_t blist;       // i32 [T*k]  bucket position -> token
  size_t hh;          // u16 [T*k][I] bf16 high part of h (k-permuted)
  size_t hl;          // u16 [T*k][I] bf16 low part of h
  size_t hsum;        // f32 [T*k][I/64]
  size_t y;           // f32 [T*k][H] per-assignment expert outputs
  size_t sh_hh;       // u16 [T][I]
  size_t sh_hl;       // u16 [T][I]
  size_t sh_hsum;     // f32 [T][I/64]
  size_t ysh;         // f32 [T][H]
  size_t total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline int gu_chunk(int H) {
  if (H % 512 == 0) return 512;
  if (H % 256 == 0) return 256;
  return 128;
}

// Upper bound of the number of sub-slots (runs of <= 8 tokens of one expert).
inline long max_subslots(long T, long E, long k) {
  const long P = T * k;
  return (E < P ? E : P) + (P + 7) / 8 + 1;
}

inline WsLayout ws_layout(long T, long E, long k, long H, long I) {
  WsLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const long P = T * k;
  const long mss = max_subslots(T, E, k);
  L.ctrl = take(16384);
  L.logits = take(4 * T * E);
  L.gate_logit = take(4 * T);
  L.xperm = take(2 * T * H);
  L.xsum = take(4 * T * (H / 64));
  L.idx = take(4 * P);
  L.w = take(4 * P);
  L.sgw = take(4 * T);
  L.offsets = take(4 * (E + 1));
  L.perm = take(4 * P);
  L.nss = take(4);
  L.ss_e = take(4 * mss);
  L.ss_off = take(4 * mss);
  L.ss_cnt = take(4 * mss);
  L.ss_rows = take(4 * 8 * mss);
  L.blist = take(4 * P);
  L.hh = take(2 * P * I);
  L.hl = take(2 * P * I);
  L.hsum = take(4 * P * (I / 64));
  L.y = take(4 * P * H);
  L.sh_hh = take(2 * T * I);
  L.sh_hl = take(2 * T * I);
  L.sh_hsum = take(4 * T * (I / 64));
  L.ysh = take(4 * T * H);
  L.total = o;
  return L;
}

// ---------------------------------------------------------------------------
// Numeric helpers.

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(uint32_t(b) << 16);
}

__device__ __forceinline__ float act_to_float(uint16_t v, bool f16) {
  return f16 ? half_bits_to_float(v) : bf16_bits_to_float(v);
}

__device__ __forceinline__ uint16_t float_to_act_bits(float v, bool f16) {
  return f16 ? __half_as_ushort(__float2half_rn(v)) : __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Ordering used by the router: a ranks before b when its logit is larger,
// equal logits by the lower id; NaN ranks below every number, NaNs by id.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  const bool na = va != va, nb = vb != vb;
  if (na != nb) return nb;
  if (!na && va != vb) return va > vb;
  return ia < ib;
}

// Storage position of k-index j inside its block of 8: the operand rows of the
// decode MMA are stored as [x0 x4 x1 x5 x2 x6 x3 x7] per block so that each
// thread's B fragment for one 64-group is 32 contiguous bytes (see
// gemv.cu, "fragment mapping").
__device__ __forceinline__ int kperm_pos(int j) {
  const int jj = j & 7;
  return (j & ~7) | (jj < 4 ? 2 * jj : 2 * (jj - 4) + 1);
}

// ---------------------------------------------------------------------------
// Warp MMA m16n8k16 with fp32 accumulation (register layouts as in the PTX ISA:
// a0 = A[g][2t..2t+1], a1 = A[g+8][2t..], a2 = A[g][2t+8..], a3 = A[g+8][2t+8..];
// b0 = B[2t..2t+1][g], b1 = B[2t+8..][g]; c0,c1 = C[g][2t..], c2,c3 = C[g+8][2t..]).
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t a0, const uint32_t a1,
                                         const uint32_t a2, const uint32_t a3, const uint32_t b0,
                                         const uint32_t b1) {
  // not volatile: a pure register operation, so the compiler may interleave
  // independent MMAs and hide their latency
  if constexpr (F16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Two 4-bit codes (bits [0,4) and [16,20) of v) -> two exact 16-bit floats.
// The code is ORed into the mantissa of 128.0 (bf16 0x4300) or 1024.0 (fp16
// 0x6400), whose last mantissa bit is worth 1, and the offset is subtracted:
// both steps are exact, so the pair holds the integer codes exactly.
template <bool F16>
__device__ __forceinline__ uint32_t codes_to_pair(uint32_t v) {
  if constexpr (F16) {
    uint32_t r = (v & 0x000F000Fu) | 0x64006400u;
    __half2 h = *reinterpret_cast<__half2*>(&r);
    const __half2 off = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    h = __hsub2(h, off);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    uint32_t r = (v & 0x000F000Fu) | 0x43004300u;
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&r);
    const __nv_bfloat162 off =
        __halves2bfloat162(__ushort_as_bfloat16(0x4300), __ushort_as_bfloat16(0x4300));
    h = __hsub2(h, off);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// 8 three-bit codes (bits [3i, 3i+3) of the low 24 bits) -> 8 nibbles
// (bits [4i, 4i+4)), so the 3-bit path feeds the same MMA operands as 4-bit.
__device__ __forceinline__ uint32_t spread3to4(uint32_t v) {
  uint32_t u = (v & 0x00000FFFu) | ((v << 4) & 0x0FFF0000u);
  u = (u & 0x003F003Fu) | ((u << 2) & 0x3F003F00u);
  u = (u & 0x07070707u) | ((u << 1) & 0x70707070u);
  return u;
}

// ---------------------------------------------------------------------------
// cp.async (LDGSTS) helpers.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src));
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(dst)), "l"(src));
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ---------------------------------------------------------------------------
// TMA bulk copies (cp.async.bulk) completing on a shared-memory mbarrier.
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
// make mbarrier inits and earlier generic shared-memory writes visible to the
// async proxy (the TMA engine)
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of a stage barrier (each try_wait suspends
// for a hardware-defined interval); false after the limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  for (int i = 0; i < (1 << 22); ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

}  // namespace moe
