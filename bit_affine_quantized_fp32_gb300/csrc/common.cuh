// common.cuh -- device helpers shared by the MoE kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

constexpr int kWarp = 32;

// Control region of a workspace (its first kCtlBytes, which
// moe_workspace_init zeroes): int32 control words, then (from byte
// kCtlTaggedOffset) the fused decode kernel's router logits, one 64-bit word
// per (token, router row) holding the call's generation number in the high
// half and the fp32 logit in the low half.
constexpr int kCtlStatus = 0;      // device status: MOE_OK or MOE_ERR_TIMEOUT
constexpr int kCtlWaitLimit = 36;  // limit of every bounded wait, microseconds (0: 1 s)
constexpr int kCtlTaggedOffset = 16384;
constexpr int kTaggedRows = 32 * 260;  // tokens x (experts + shared gate), rounded
constexpr int kCtlBytes = kCtlTaggedOffset + 8 * kTaggedRows;

// ---------------------------------------------------------------------------
// Workspace layout.  Every region is 256-byte aligned; the layout depends only
// on the call's shape, so any workspace of moe_workspace_bytes(max_tokens, ...)
// bytes serves every call with n_tokens <= max_tokens.  Sums are kept in the
// padded per-chunk layout of engine.cuh (ldx / ldh floats per row).
struct WsLayout {
  size_t ctrl;        // control region (kCtlBytes): words, tagged logits
  size_t logits;      // f32 [T][E]
  size_t gate_logit;  // f32 [T]
  size_t idx;         // i32 [T][k]
  size_t w;           // f32 [T][k]
  size_t sgw;         // f32 [T]
  size_t offsets;     // i32 [E+1]
  size_t perm;        // i32 [T*k]
  size_t nss;         // i32 [1]   number of sub-slots
  size_t ss_e;        // i32 [maxss] expert of each sub-slot
  size_t ss_off;      // i32 [maxss] first bucket position
  size_t ss_cnt;      // i32 [maxss] tokens (1..8)
  size_t xsum;        // f32 [T][ldx] per-64-group sums of x
  size_t hh;          // u16 [T*k][I+8] bf16 high part of h (padded pitch)
  size_t hl;          // u16 [T*k][I+8] bf16 low part of h
  size_t hsum;        // f32 [T*k][ldh]
  size_t y;           // f32 [2][T*k][H] per-assignment expert outputs (k-half planes)
  size_t sh_hh;       // u16 [T][I+8]
  size_t sh_hl;       // u16 [T][I+8]
  size_t sh_hsum;     // f32 [T][ldh]
  size_t ysh;         // f32 [2][T][H]
  size_t pt_n;        // i32 [1]   prefill tiles (experts with many assignments)
  size_t pt_e;        // i32 [maxss] expert of each tile
  size_t pt_off;      // i32 [maxss] first bucket position
  size_t pt_cnt;      // i32 [maxss] rows (1..128)
  size_t xh;          // u16 [T][H] fp16 copy of bf16 activations (prefill form)
  size_t rpart;       // f32 [4][T][E+1] k-slice sums of the router (prefill form)
  size_t rsplit;      // u16 [3][E+1][H] + [2][T][H] bf16 parts of the router rows and of
                      //     fp16 x (prefill form)
  size_t total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Upper bound of the number of sub-slots (runs of <= 8 tokens of one expert).
inline long max_subslots(long T, long E, long k) {
  const long P = T * k;
  return (E < P ? E : P) + (P + 7) / 8 + 1;
}

// floats per row of the padded sums of a K-wide operand (see engine.cuh)
inline long padded_sums_ld(long K) {
  const long CK = K % 512 == 0 ? 512 : (K % 256 == 0 ? 256 : 128);
  return (K / CK) * (((CK / 64) + 3) & ~3L);
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
  const long ldx = padded_sums_ld(H), ldh = padded_sums_ld(I);
  L.ctrl = take(kCtlBytes);
  L.logits = take(4 * T * E);
  L.gate_logit = take(4 * T);
  L.idx = take(4 * P);
  L.w = take(4 * P);
  L.sgw = take(4 * T);
  L.offsets = take(4 * (E + 1));
  L.perm = take(4 * P);
  L.nss = take(4);
  L.ss_e = take(4 * mss);
  L.ss_off = take(4 * mss);
  L.ss_cnt = take(4 * mss);
  L.xsum = take(4 * T * ldx);
  L.hh = take(2 * P * (I + 8));   // rows at a pitch of I + 8 elements
  L.hl = take(2 * P * (I + 8));
  L.hsum = take(4 * P * ldh);
  L.y = take(4 * 2 * P * H);     // two k-half planes
  L.sh_hh = take(2 * T * (I + 8));
  L.sh_hl = take(2 * T * (I + 8));
  L.sh_hsum = take(4 * T * ldh);
  L.ysh = take(4 * 2 * T * H);
  L.pt_n = take(4);
  L.pt_e = take(4 * mss);
  L.pt_off = take(4 * mss);
  L.pt_cnt = take(4 * mss);
  L.xh = take(2 * T * H);
  L.rpart = take(4 * 4 * T * (E + 1));
  L.rsplit = take(2 * (3 * (E + 1) * H + 2 * T * H));
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

// v rounded to bf16 (nearest, ties to even) and widened back to fp32.
__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
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

// ---------------------------------------------------------------------------
// cp.async (LDGSTS) helpers.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src));
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
// Bring `bytes` (a multiple of 16, 16-byte aligned) at src into L2 ahead of
// a later copy, without waiting for it.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
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
