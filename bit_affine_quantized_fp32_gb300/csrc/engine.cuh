// engine.cuh -- the warp-specialised item engine of the decode path, shared
// by the standalone expert kernels (units.cu) and the fused layer kernel
// (decode.cu).
//
// A CTA has 19 warps: warps 0..15 are the consumers, warp 16 the producer
// (weights), warp 17 the operand warp, warp 18 the signal warp.
// Work comes as "units": one sub-slot (<= 8 tokens of one expert) times one
// 128-row block of a matrix, streamed as k-chunk "items".  An item is a
// contiguous block of the kernel-tiled bank (codes + scales, tiled.cuh); the
// unit's operand rows (x, or h as bf16 hi + lo, full K) and their per-64-group
// sums sit in one of two operand buffers for the whole unit.
//   producer: claims units from the schedule (a queue shared by the grid in
//             the fused kernel), publishes each into a ring of unit
//             descriptors in shared memory, and streams its weight items by
//             TMA bulk copy into the stage ring (waiting only until a stage
//             is free), so weights keep flowing while operands wait;
//   operand:  per unit, waits for the unit's dependency on other CTAs (h
//             rows, y rows for a combine piece) if any, then fills an operand
//             buffer (one copy per x row, or three block copies for h);
//   consumers: wait for the operand buffer and each item's stage, run the MMA
//             pass, release the stage, and after the last item reduce and
//             write the unit's result (SwiGLU -> h, or y);
//   signal:   publishes finished units to other CTAs with a release
//             reduction, so no consumer waits on a gpu-scope release.
// There is no CTA-wide barrier in the unit loop; consumers synchronise only
// among themselves in a unit's epilogue.
//
// Warp w of the consumers owns the 16-row M-tile (w & 7) and the k-half
// (w >> 3) of every chunk; the two halves are added in a fixed order at the
// end of a unit.  Arithmetic per weight row r, 64-code group G and token n:
//   sum_i (s q_i + b) x_i = s * (sum_i q_i x_i) + b * X_G(n)
// The bracket is an mma.sync m16n8k16 with the codes as exact bf16/fp16
// integers (fp32 accumulation, exact products); s and b are applied in fp32.
// Every output element is one MMA column with a fixed k-order and fixed fp32
// reductions, so a token's result never depends on the other tokens of the
// call, on its sub-slot or on the CTA that runs the unit, and the fused and
// standalone kernels (same device functions) give the same bits.
//
// Source: "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803",
// comment "Progress on the 4-bit gate" (grouped affine experts with a SwiGLU
// epilogue, decode rows summed in fp32); "Native server: --backend xpu for
// Nemotron on Intel Arc", update comment (expert reads shared across rows).
#pragma once

#include "common.cuh"
#include "tiled.cuh"

namespace moe {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;     // 512
constexpr int kProducerWarp = kConsumerWarps;       // weights
constexpr int kOperandWarp = kConsumerWarps + 1;    // operand rows
constexpr int kSignalWarp = kConsumerWarps + 2;     // publishes finished units
constexpr int kEngineThreads = kConsumers + 96;
constexpr int kUnitRing = 16;                       // unit descriptors in flight
constexpr int kRingReaders = kConsumerWarps + 2;    // consumer, operand and signal warps
constexpr int kEpiRing = 4;
constexpr int kUnitRows = 128;
constexpr int kMaxTok = 8;
constexpr int kMaxStages = 6;
constexpr int kEngineSmemMax = 227 * 1024;

__host__ __device__ inline int align16i(int x) { return (x + 15) & ~15; }
__host__ __device__ inline int align128i(int x) { return (x + 127) & ~127; }
__host__ __device__ inline int round4(int x) { return (x + 3) & ~3; }

// A matrix family (w13 or w2) of a tiled bank.
struct MatGeo {
  TileGeo t;
  const uint8_t* base;  // tiled buffer (expert 0, item 0)
};

// Padded per-token sums of an operand: 64-group j of a row of K values sits at
// (j / ng) * ngp + j % ng with ng = CK / 64 and ngp = ng rounded up to 4, so
// each chunk's sums start on a 16-byte boundary (one bulk copy per row).
__host__ __device__ inline int sums_ngp(const TileGeo& t) { return round4(t.ng); }
__host__ __device__ inline int sums_ld(const TileGeo& t) { return t.nch * sums_ngp(t); }
__host__ __device__ inline int sums_pos(const TileGeo& t, int j) {
  return (j / t.ng) * sums_ngp(t) + j % t.ng;
}

// A unit covers a 128-row block (gate/up: 64 gate rows + their 64 up rows);
// the consumers split it as 8 M-tiles x 2 groups of k.
constexpr int kTiles = 8, kKsplit = 2;



enum : int { kItemGateUp = 0, kItemDown = 1, kItemCombine = 2, kItemEnd = 3 };

// A weight stage holds one tiled item.
__host__ __device__ inline int stage_bytes(const TileGeo& t) { return align128i(t.item_bytes); }

// Operand buffer of a unit: [rows hi][rows lo (split operands)][sums], rows of
// the full K at a pitch 16 bytes past a multiple of 128 (conflict-free
// fragment loads), sums rows of sums_ld(t) floats.
struct OpLayout {
  int x, xlo, xs, bpitch, lds, bytes;
};

__host__ __device__ inline OpLayout op_layout(const TileGeo& t) {
  OpLayout L;
  L.bpitch = t.K * 2 + 16;
  L.lds = sums_ld(t);
  L.x = 0;
  L.xlo = kMaxTok * L.bpitch;
  L.xs = t.down ? 2 * kMaxTok * L.bpitch : L.xlo;
  L.bytes = align128i(L.xs + kMaxTok * L.lds * 4);
  return L;
}

// Where the consumers' results go, per matrix slot.
struct MatTarget {
  uint16_t* hh;   // gate/up: h hi part [rows][I + 8] (bf16, padded pitch)
  uint16_t* hl;   //          h lo part
  float* hsum;    //          padded sums of hi + lo per 64-group
  float* hout;    //          nullable fp32 h [rows][I]
  float* y;       // down:    [2][rows][H] fp32, one plane per k-half
  size_t yhalf;   //          elements from the first plane to the second
};

// Row pitch (elements) of h in the workspace: 16 bytes past the row, so that a
// run of consecutive rows copies straight into an operand buffer.
__host__ __device__ inline int h_pitch(int I) { return I + 8; }

struct EngineCfg {
  MatGeo geo[4];
  MatTarget tg[4];
  int inter, hidden;
  int* status;     // device status word
  uint32_t magic_bf16;  // 0x43004300, see code_pair (held in the parameter space
  uint32_t magic_f16;   // 0x64006400  so the compiler keeps it out of immediates)
};

// ---------------------------------------------------------------------------
// Barrier helpers (all waits bounded).

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
  return t;
}

// try_wait that lets the thread sleep (up to `hint_ns`) until the phase
// completes instead of spinning
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, unsigned parity,
                                                    unsigned hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // default: one second
constexpr unsigned long long kDrainLimitNs = 100000000ull;  // copies in flight at exit

// Bounded-wait control of one CTA (shared memory): the limit of every wait,
// read once at kernel start from the workspace control word kCtlWaitLimit
// (microseconds; 0 selects the one-second default), and the flag set after
// the first timeout, which turns every later wait of the CTA into a no-op so
// that the kernel finishes (with garbage results) quickly.
struct WaitCtl {
  unsigned long long limit_ns;
  int skip;
};

// One thread; `ctrl` is the workspace's control region (nullable: default).
__device__ __forceinline__ void wait_ctl_init(WaitCtl& w, const int* ctrl) {
  const int us = ctrl ? *(volatile const int*)(ctrl + kCtlWaitLimit) : 0;
  w.limit_ns = us > 0 ? 1000ull * unsigned(us) : kWaitLimitNs;
  w.skip = 0;
}

// Wait for phase `parity` of an mbarrier; after the CTA's limit, record a
// timeout and return false.  By default the warp polls (the decode engine's
// waits are short and a suspended warp wakes late); sleep = true lets the
// hardware suspend it between polls (long waits of otherwise idle roles).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity, WaitCtl* w,
                                                  int* status, bool sleep = false) {
  auto poll = [&]() {
    return sleep ? mbar_try_wait_sleep(bar, parity, 100000u) : mbar_try_wait(bar, parity);
  };
  if (poll()) return true;
  volatile int* skip = &w->skip;
  const unsigned long long t0 = global_ns(), lim = w->limit_ns;
  for (;;) {
    if (poll()) return true;
    if (*skip) return false;
    if (global_ns() - t0 > lim) break;
  }
  *skip = 1;
  atomicExch(status, int(MOE_ERR_TIMEOUT));
  return false;
}

// Wait for the completion of a copy this CTA issued (its barrier phase
// `parity`) before the CTA exits; unlike the other waits it does not give up
// after a timeout elsewhere in the CTA, only after kDrainLimitNs.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 10000u)) return true;
    if (global_ns() - t0 > kDrainLimitNs) return false;
  }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// add `bytes` to the current phase's expected transaction count (no arrival)
__device__ __forceinline__ void mbar_expect_only(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// the consumers' own barrier (named barrier 1, 512 threads)
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kConsumers) : "memory");
}

// order data acquired through the generic proxy before later TMA reads
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// two consecutive 64-bit words (16-byte aligned), each read single-copy atomically
__device__ __forceinline__ void ld_relaxed_v2u64(const unsigned long long* p, unsigned long long& a,
                                                 unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];\n"
               : "=l"(a), "=l"(b)
               : "l"(p)
               : "memory");
}

__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait (one thread) until *p >= target; after the CTA's limit records
// a timeout and sets the skip flag.  Returns at once when the flag is set.
static __device__ __noinline__ bool wait_counter(const int* p, int target, WaitCtl* w,
                                                 int* status) {
  if (ld_acquire(p) >= target) return true;
  volatile int* skip = &w->skip;
  const unsigned long long t0 = global_ns(), lim = w->limit_ns;
  unsigned ns = 32;
  for (;;) {
    if (ld_acquire(p) >= target) return true;
    if (*skip) return false;
    if (global_ns() - t0 > lim) break;
    __nanosleep(ns);
    if (ns < 64) ns <<= 1;
  }
  *skip = 1;
  atomicExch(status, int(MOE_ERR_TIMEOUT));
  return false;
}

}  // namespace moe

namespace moe {

// ---------------------------------------------------------------------------
// Consumer arithmetic.

// Two codes (bits [0,4) and [16,20) of v) -> two 16-bit floats: one lop3
// (v & 0x000F000F) | magic.  bf16: magic 0x43004300 (128.0) gives exactly
// 128 + q; the 128 is taken out in the fold (bias' = bias - 128 scale).
// fp16: magic 0x64006400 (1024.0) gives 1024 + q, minus 1024 exactly.  The
// magic comes in a register (a kernel parameter): with both constants as
// immediates the compiler emits two instructions, and the code conversion is
// what bounds the consumers (integer ALU pipe).
template <bool F16>
__device__ __forceinline__ uint32_t code_pair(uint32_t v, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;\n" : "=r"(r) : "r"(v), "r"(magic));
  if constexpr (F16) {
    __half2 h = *reinterpret_cast<__half2*>(&r);
    const __half2 off = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    h = __hsub2(h, off);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    return r;
  }
}

// code_pair with the pair's high bits (at [4,6) and [20,22)) added: codes up
// to 6 bits stay exact (bf16 128 + q for q < 128, fp16 1024 + q).
template <bool F16A>
__device__ __forceinline__ uint32_t code_pair_hb(uint32_t v, uint32_t hb, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;\n" : "=r"(r) : "r"(v), "r"(hb | magic));
  if constexpr (F16A) {
    __half2 h = *reinterpret_cast<__half2*>(&r);
    const __half2 off = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    h = __hsub2(h, off);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    return r;
  }
}

// Two nibbles as the exact 16-bit values q (no +128 offset): the high nibble
// pair of an 8-bit code, whose second MMA is scaled by 16.
template <bool F16A>
__device__ __forceinline__ uint32_t code_pair_exact(uint32_t v, uint32_t magic) {
  uint32_t r = code_pair<F16A>(v, magic);
  if constexpr (!F16A) {
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&r);
    const __nv_bfloat162 off = __halves2bfloat162(__ushort_as_bfloat16(0x4300),
                                                  __ushort_as_bfloat16(0x4300));
    b = __hsub2(b, off);
    r = *reinterpret_cast<uint32_t*>(&b);
  }
  return r;
}

// shift right by s (left by -s), s a compile-time constant after inlining
__device__ __forceinline__ uint32_t shr_signed(uint32_t v, int s) { return s >= 0 ? v >> s : v << -s; }

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t v) {
  return __half22float2(*reinterpret_cast<__half2*>(&v));
}

// One k-chunk item (chunk c) for consumer warp (tile, ks): the item's stage
// holds TILES M-tiles (codes: tile t, group G at (t * NG + G) * CB; then the
// scales of the TILES tiles), and the warp takes the groups G = ks, ks +
// KSPLIT, ... < NG of its tile, added into acc.  NG = CK/64 is a compile-time
// constant so the group loop unrolls completely (a rolled loop costs several
// times the instructions).  op is the unit's operand buffer.  acc[0]: (row g,
// token 2t), acc[1]: (g, 2t+1), acc[2]: (g+8, 2t), acc[3]: (g+8, 2t+1).
// Operand columns of tokens >= cnt hold whatever the buffer held before; MMA
// columns are independent, so they only touch accumulators that are never
// written out.
template <int FMT, bool F16A, bool SPLIT, int NG, int TILES, int KSPLIT>
__device__ __forceinline__ void compute_item(const TileGeo& tg, const uint8_t* wst,
                                             const uint8_t* op, const OpLayout& L, int c,
                                             int tile, int ks, uint32_t mg, float (&acc)[4]) {
  constexpr int CB = tiled_cb(FMT);
  constexpr int BITS = tiled_bits(FMT);
  constexpr int NGP = (NG + 3) & ~3;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;
  const int xo = gq * L.bpitch + c * NG * 128 + 32 * t;
  const uint8_t* xrow = op + L.x + xo;
  const uint8_t* xlrow = op + L.xlo + xo;
  const float* xs0 = reinterpret_cast<const float*>(op + L.xs) + (2 * t) * L.lds + c * NGP;
  const float* xs1 = xs0 + L.lds;
  const uint8_t* sc = wst + TILES * NG * CB;
#pragma unroll
  for (int i = 0; i < (NG + KSPLIT - 1) / KSPLIT; ++i) {
    const int G = ks + KSPLIT * i;
    if (NG % KSPLIT != 0 && G >= NG) break;
    const uint8_t* codes = wst + (tile * NG + G) * CB;
    // the lane's four nibble words (low 4 bits of its 32 codes) and what
    // the format keeps above them
    uint32_t w[4], hw[4] = {0u, 0u, 0u, 0u}, p0 = 0u, p1 = 0u;
    if constexpr (BITS <= 3) {
      const uint32_t* pl = reinterpret_cast<const uint32_t*>(codes) + lane;
      planes_to_words(pl[0], pl[32], BITS == 3 ? pl[64] : 0u, w[0], w[1], w[2], w[3]);
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(codes + lane * 16);
      w[0] = v.x;
      w[1] = v.y;
      w[2] = v.z;
      w[3] = v.w;
      if constexpr (BITS == 5 || BITS == 6) {
        const uint32_t* hp = reinterpret_cast<const uint32_t*>(codes + 512) + lane;
        p0 = hp[0];
        if constexpr (BITS == 6) p1 = hp[32];
      } else if constexpr (BITS == 8) {
        const uint4 h = *reinterpret_cast<const uint4*>(codes + 512 + lane * 16);
        hw[0] = h.x;
        hw[1] = h.y;
        hw[2] = h.z;
        hw[3] = h.w;
      }
    }
    // the code pair in nibbles m and m + 4 of word x, as an MMA register
    auto pr = [&](int x, int m) -> uint32_t {
      const uint32_t v = w[x] >> (4 * m);
      if constexpr (BITS == 5) {
        return code_pair_hb<F16A>(v, shr_signed(p0, 4 * x + m - 4) & 0x00100010u, mg);
      } else if constexpr (BITS == 6) {
        return code_pair_hb<F16A>(
            v, shr_signed(x < 2 ? p0 : p1, 2 * (4 * (x & 1) + m) - 4) & 0x00300030u, mg);
      } else {
        return code_pair<F16A>(v, mg);
      }
    };
    const uint4 xa = *reinterpret_cast<const uint4*>(xrow + G * 128);
    const uint4 xb = *reinterpret_cast<const uint4*>(xrow + G * 128 + 16);
    // k-step m takes code pairs (4m, 4m+1) and (4m+2, 4m+3) of the lane's 16
    // codes: nibbles (m&1)*2 and (m&1)*2+1 of word W0/W1 (row g), W2/W3 (g+8)
    const uint32_t A00 = pr(0, 0), A01 = pr(2, 0), A02 = pr(0, 1), A03 = pr(2, 1);
    const uint32_t A10 = pr(0, 2), A11 = pr(2, 2), A12 = pr(0, 3), A13 = pr(2, 3);
    const uint32_t A20 = pr(1, 0), A21 = pr(3, 0), A22 = pr(1, 1), A23 = pr(3, 1);
    const uint32_t A30 = pr(1, 2), A31 = pr(3, 2), A32 = pr(1, 3), A33 = pr(3, 3);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma16816<F16A>(d, A00, A01, A02, A03, xa.x, xa.y);
    mma16816<F16A>(d, A10, A11, A12, A13, xa.z, xa.w);
    mma16816<F16A>(d, A20, A21, A22, A23, xb.x, xb.y);
    mma16816<F16A>(d, A30, A31, A32, A33, xb.z, xb.w);
    if constexpr (SPLIT) {
      const uint4 la = *reinterpret_cast<const uint4*>(xlrow + G * 128);
      const uint4 lb = *reinterpret_cast<const uint4*>(xlrow + G * 128 + 16);
      mma16816<F16A>(d, A00, A01, A02, A03, la.x, la.y);
      mma16816<F16A>(d, A10, A11, A12, A13, la.z, la.w);
      mma16816<F16A>(d, A20, A21, A22, A23, lb.x, lb.y);
      mma16816<F16A>(d, A30, A31, A32, A33, lb.z, lb.w);
    }
    if constexpr (BITS == 8) {
      // the high nibbles as exact values: q = lo + 16 hi, so the group's
      // bracket is d_lo + 16 d_hi
      auto hp = [&](int x, int m) -> uint32_t { return code_pair_exact<F16A>(hw[x] >> (4 * m), mg); };
      float dh[4] = {0.f, 0.f, 0.f, 0.f};
      mma16816<F16A>(dh, hp(0, 0), hp(2, 0), hp(0, 1), hp(2, 1), xa.x, xa.y);
      mma16816<F16A>(dh, hp(0, 2), hp(2, 2), hp(0, 3), hp(2, 3), xa.z, xa.w);
      mma16816<F16A>(dh, hp(1, 0), hp(3, 0), hp(1, 1), hp(3, 1), xb.x, xb.y);
      mma16816<F16A>(dh, hp(1, 2), hp(3, 2), hp(1, 3), hp(3, 3), xb.z, xb.w);
      if constexpr (SPLIT) {
        const uint4 la = *reinterpret_cast<const uint4*>(xlrow + G * 128);
        const uint4 lb = *reinterpret_cast<const uint4*>(xlrow + G * 128 + 16);
        mma16816<F16A>(dh, hp(0, 0), hp(2, 0), hp(0, 1), hp(2, 1), la.x, la.y);
        mma16816<F16A>(dh, hp(0, 2), hp(2, 2), hp(0, 3), hp(2, 3), la.z, la.w);
        mma16816<F16A>(dh, hp(1, 0), hp(3, 0), hp(1, 1), hp(3, 1), lb.x, lb.y);
        mma16816<F16A>(dh, hp(1, 2), hp(3, 2), hp(1, 3), hp(3, 3), lb.z, lb.w);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) d[q] = fmaf(16.f, dh[q], d[q]);
    }
    float s0, s1, b0, b1;
    if constexpr (FMT == MOE_FMT_W4A16_SYM_G128) {
      const uint32_t sv =
          *reinterpret_cast<const uint32_t*>(sc + ((tile * 8 + gq) * (NG / 2) + (G >> 1)) * 4);
      const float2 sf = half2_bits_to_float2(sv);
      s0 = sf.x;
      s1 = sf.y;
      // w = s (u - 8) for the stored nibble u; with the bf16 operand's +128
      // the offset is -136 s (exact: an fp16 times 136 fits in fp32)
      b0 = (F16A ? -8.f : -136.f) * s0;
      b1 = (F16A ? -8.f : -136.f) * s1;
    } else {
      const uint2 sv = *reinterpret_cast<const uint2*>(sc + ((tile * 8 + gq) * NG + G) * 8);
      const float2 p0 = half2_bits_to_float2(sv.x), p1 = half2_bits_to_float2(sv.y);
      s0 = p0.x;
      b0 = p0.y;
      s1 = p1.x;
      b1 = p1.y;
      if constexpr (!F16A) {  // operand codes carry +128
        b0 = fmaf(-128.f, s0, b0);
        b1 = fmaf(-128.f, s1, b1);
      }
    }
    const float X0 = xs0[G], X1 = xs1[G];
    acc[0] = fmaf(s0, d[0], acc[0]);
    acc[0] = fmaf(b0, X0, acc[0]);
    acc[1] = fmaf(s0, d[1], acc[1]);
    acc[1] = fmaf(b0, X1, acc[1]);
    acc[2] = fmaf(s1, d[2], acc[2]);
    acc[2] = fmaf(b1, X0, acc[2]);
    acc[3] = fmaf(s1, d[3], acc[3]);
    acc[3] = fmaf(b1, X1, acc[3]);
  }
}

}  // namespace moe

namespace moe {

// ---------------------------------------------------------------------------
// Units and where their rows come from / go to.

// Operand source of a matrix slot: rows of B (and Blo) at a pitch of ldB
// elements and their padded per-64-group sums (row stride ldS floats).
// block = 1: the rows of a unit are consecutive and ldB*2 equals the operand
// buffer's pitch (h in the workspace), so each part is one bulk copy;
// block = 0: one copy per row (x rows, gathered by token).
struct MatSource {
  const uint16_t* B;
  const uint16_t* Blo;  // nullptr unless the operand is split (h)
  const float* Bsum;
  int ldB, ldS, block;
};

enum : int {
  kRowsDirect = 0,  // operand row = output row = off + n (tokens of a fixed expert)
  kRowsGather = 1,  // operand row = perm[off + n] / k (token), output row = off + n
  kRowsScatter = 2  // operand row = off + n, output row = perm[off + n] (assignment)
};

struct UnitInfo {
  int kind;         // kItemGateUp, kItemDown or kItemCombine
  int mat;          // matrix slot
  int e, blk, off, cnt, nch;
  int rows;         // kRows*
  int signal;       // control word += 1 after the epilogue, -1 for none
  int wait_ctr;     // control word the operands wait for (-1: none)
  int wait_target;
};

__device__ __forceinline__ int unit_op_row(const UnitInfo& u, const int* perm, int k, int n) {
  if (u.rows == kRowsGather) return perm[u.off + n] / k;
  return u.off + n;
}

__device__ __forceinline__ int unit_out_row(const UnitInfo& u, const int* perm, int n) {
  if (u.rows == kRowsScatter) return perm[u.off + n];
  return u.off + n;
}

// Engine shared memory (static part).
struct EngineSmem {
  uint64_t full[kMaxStages];      // weight stages
  uint64_t empty[kMaxStages];
  uint64_t op_full[2];            // operand buffers
  uint64_t op_empty[2];
  uint64_t epi_full[kEpiRing];    // unit results written (consumers -> signal warp)
  uint64_t epi_empty[kEpiRing];   // unit published (signal warp -> consumers)
  uint64_t ring_full[kUnitRing];  // unit descriptor published (producer -> readers)
  uint64_t ring_empty[kUnitRing]; // descriptor read by every reader warp
  UnitInfo ring[kUnitRing];
  WaitCtl wc;                     // wait limit and timeout flag
  float red[2][8][32][4];         // epilogue: accumulators by k-half, tile, lane
  float part[kConsumerWarps];     // epilogue: per-warp partial sums
};

// `ctrl`: the workspace's control region (the wait limit).
__device__ __forceinline__ void engine_init(EngineSmem& E, int S, const int* ctrl) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&E.full[s], 1);
      mbar_init(&E.empty[s], kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&E.op_full[b], 1);
      mbar_init(&E.op_empty[b], kConsumerWarps);
    }
    for (int b = 0; b < kEpiRing; ++b) {
      mbar_init(&E.epi_full[b], kConsumerWarps);
      mbar_init(&E.epi_empty[b], 1);
    }
    for (int b = 0; b < kUnitRing; ++b) {
      mbar_init(&E.ring_full[b], 1);
      mbar_init(&E.ring_empty[b], kRingReaders);
    }
    wait_ctl_init(E.wc, ctrl);
  }
}

// Dynamic shared memory of the engine: nob operand buffers of OB bytes, then
// S weight stages of SB bytes.
struct EngineMem {
  uint8_t* ops;
  uint8_t* stages;
  int OB, nob, SB, S;
};

// Ring position: slot and how many times it has been used.
struct Ring {
  int slot, use, S;
  __device__ void next() {
    if (++slot == S) {
      slot = 0;
      ++use;
    }
  }
};

// ---------------------------------------------------------------------------
// A unit's MMA pass: wait for the operand buffer, then for every k-chunk wait
// for its stage, run compute_item and release the stage.  The format, group
// count, operand split and warp split are resolved once per unit (unit_mat),
// so the chunk loop carries no per-item dispatch or layout arithmetic.  Warp
// w takes M-tile w % 8 and k-group w / 8.
template <int FMT, bool F16A, bool SPLIT, int NG>
__device__ __forceinline__ void unit_items(const TileGeo& tg, uint32_t mg, EngineSmem& E,
                                           const EngineMem& M, Ring& R, const uint8_t* op,
                                           uint64_t* op_full, unsigned op_parity, int* status,
                                           float (&acc)[4]) {
  const int warp = threadIdx.x >> 5;
  const int tile = warp % kTiles, ks = warp / kTiles;
  const OpLayout L = op_layout(tg);
  const int nch = tg.nch;
  mbar_wait_bounded(op_full, op_parity, &E.wc, status);
  for (int c = 0; c < nch; ++c) {
    mbar_wait_bounded(&E.full[R.slot], R.use & 1, &E.wc, status);
    compute_item<FMT, F16A, SPLIT, NG, kTiles, kKsplit>(tg, M.stages + (size_t)R.slot * M.SB, op,
                                                        L, c, tile, ks, mg, acc);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&E.empty[R.slot]);
    R.next();
  }
}

template <int FMT, bool F16A, bool SPLIT>
__device__ __forceinline__ void unit_ng(const TileGeo& tg, uint32_t mg, EngineSmem& E,
                                        const EngineMem& M, Ring& R, const uint8_t* op,
                                        uint64_t* op_full, unsigned op_parity, int* status,
                                        float (&acc)[4]) {
  if (tg.ng == 8)
    unit_items<FMT, F16A, SPLIT, 8>(tg, mg, E, M, R, op, op_full, op_parity, status, acc);
  else if (tg.ng == 4)
    unit_items<FMT, F16A, SPLIT, 4>(tg, mg, E, M, R, op, op_full, op_parity, status, acc);
  else
    unit_items<FMT, F16A, SPLIT, 2>(tg, mg, E, M, R, op, op_full, op_parity, status, acc);
}

// Matrix slot `mat` (0/2 gate/up, 1/3 down); slots 0/1 hold format FMT,
// slots 2/3 format FMT_SH (with FMT_SH == FMT both share one copy of the
// code).  The down operand (h) is split bf16 whatever the activation type.
template <int FMT, int FMT_SH, bool F16A>
__device__ __forceinline__ void unit_mat(const EngineCfg& C, int mat, EngineSmem& E,
                                         const EngineMem& M, Ring& R, const uint8_t* op,
                                         uint64_t* op_full, unsigned op_parity,
                                         float (&acc)[4]) {
  const TileGeo& tg = C.geo[mat].t;
  const bool down = mat & 1;
  const uint32_t mg = (F16A && !down) ? C.magic_f16 : C.magic_bf16;
  if (FMT_SH == FMT || mat < 2) {
    if (down)
      unit_ng<FMT, false, true>(tg, mg, E, M, R, op, op_full, op_parity, C.status, acc);
    else
      unit_ng<FMT, F16A, false>(tg, mg, E, M, R, op, op_full, op_parity, C.status, acc);
  } else {
    if (down)
      unit_ng<FMT_SH, false, true>(tg, mg, E, M, R, op, op_full, op_parity, C.status, acc);
    else
      unit_ng<FMT_SH, F16A, false>(tg, mg, E, M, R, op, op_full, op_parity, C.status, acc);
  }
}

// ---------------------------------------------------------------------------
// The unit ring: the producer publishes unit descriptors in claim order; the
// consumer, operand and signal warps read them in the same order.
//
// A schedule (Sched) provides
//   claim(n)    the queue index of this CTA's n-th claim (producer lane 0);
//   unit(j, u)  the unit at queue index j, false past the end;
//   source(mat), perm(), topk(), combine(blk).

__device__ __forceinline__ void ring_put(EngineSmem& E, int pos, const UnitInfo& u,
                                         int* status) {
  const int s = pos % kUnitRing;
  if (pos >= kUnitRing)
    mbar_wait_bounded(&E.ring_empty[s], ((pos / kUnitRing) - 1) & 1, &E.wc, status);
  E.ring[s] = u;
  mbar_arrive(&E.ring_full[s]);  // release: the descriptor is visible to the readers
}

// The unit at ring position pos (every lane of a reader warp); after a
// timeout the reader ends its loop (kItemEnd).
__device__ __forceinline__ UnitInfo ring_take(EngineSmem& E, int pos, int* status) {
  const int s = pos % kUnitRing;
  UnitInfo u;
  if (mbar_wait_bounded(&E.ring_full[s], (pos / kUnitRing) & 1, &E.wc, status)) {
    u = E.ring[s];
  } else {
    u = UnitInfo{};
    u.kind = kItemEnd;
  }
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&E.ring_empty[s]);
  return u;
}

// ---------------------------------------------------------------------------
// Producer (warp kProducerWarp, all 32 lanes).

// Weight item (u, c) into a stage: one bulk copy.
__device__ __forceinline__ const uint8_t* item_src(const MatGeo& g, const UnitInfo& u, int c) {
  return g.base + (size_t)u.e * g.t.expert_bytes + (size_t)(u.blk * g.t.nch + c) * g.t.item_bytes;
}

__device__ __forceinline__ void produce_weights(const MatGeo& g, const UnitInfo& u, int c,
                                                uint8_t* st, uint64_t* full) {
  if ((threadIdx.x & 31) == 0) {
    const unsigned bytes = unsigned(g.t.item_bytes);
    mbar_expect_tx(full, bytes);
    bulk_g2s(st, item_src(g, u, c), bytes, full);
  }
}

// The unit's operand rows and sums into an operand buffer, after the unit's
// dependency (if any).  Completes on *full.
__device__ __forceinline__ void produce_operands(const EngineCfg& C, const MatSource& src,
                                                 const UnitInfo& u, const int* perm, int k,
                                                 uint8_t* ob, uint64_t* full, const int* ctrl,
                                                 WaitCtl* wc) {
  const int lane = threadIdx.x & 31;
  const TileGeo& tg = C.geo[u.mat].t;
  const OpLayout L = op_layout(tg);
  if (u.wait_ctr >= 0) {
    if (lane == 0) wait_counter(ctrl + u.wait_ctr, u.wait_target, wc, C.status);
    __syncwarp();
    fence_proxy_async_global();
  }
  if (src.block) {
    const unsigned rb = unsigned(u.cnt * L.bpitch), sb = unsigned(u.cnt * L.lds * 4);
    if (lane == 0) {
      mbar_expect_tx(full, rb * (src.Blo ? 2u : 1u) + sb);
      bulk_g2s(ob + L.x, src.B + (size_t)u.off * src.ldB, rb, full);
      if (src.Blo) bulk_g2s(ob + L.xlo, src.Blo + (size_t)u.off * src.ldB, rb, full);
      bulk_g2s(ob + L.xs, src.Bsum + (size_t)u.off * src.ldS, sb, full);
    }
  } else {
    if (lane == 0) mbar_expect_only(full, unsigned(u.cnt * (tg.K * 2 + L.lds * 4)));
    __syncwarp();
    const int n = lane & 7;
    if (n < u.cnt && lane < 16) {
      const int row = unit_op_row(u, perm, k, n);
      if (lane < 8)
        bulk_g2s(ob + L.x + n * L.bpitch, src.B + (size_t)row * src.ldB, unsigned(tg.K * 2),
                 full);
      else
        bulk_g2s(ob + L.xs + n * L.lds * 4, src.Bsum + (size_t)row * src.ldS,
                 unsigned(L.lds * 4), full);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(full);
  }
}

// Items [c0, nch) of unit u into L2 (one thread), so that their later copies
// into a stage come from L2.
__device__ __forceinline__ void prefetch_unit(const EngineCfg& C, const UnitInfo& u, int c0) {
  if (u.kind != kItemGateUp && u.kind != kItemDown) return;
  const MatGeo& g = C.geo[u.mat];
  for (int c = c0; c < u.nch; ++c) bulk_prefetch_l2(item_src(g, u, c), unsigned(g.t.item_bytes));
}

// Where the producer starts: its first claimed queue index, and how many of
// that unit's weight items it already issued into stages 0.. (the fused
// kernel fills the stages with a routing-independent unit before routing).
struct ProducerStart {
  int j;
  int issued;
};

// The producer's loop: publish the unit, claim the next one (the atomic is in
// flight while this unit's items are issued), stream this unit's weight items
// into the stage ring, then prefetch the next unit's items into L2 -- which
// keeps enough bytes in flight for HBM (the stage ring alone holds too few)
// without queueing copies that are needed now behind prefetches.  The call's
// very first copy is left to land before the rest of the first unit's stages
// go out: every CTA starts at once, and a CTA's first item would otherwise
// share HBM with all the grid's later stages and land with them.
template <class Sched>
__device__ void producer_run(const EngineCfg& C, EngineSmem& E, const EngineMem& M,
                             const Sched& sch, ProducerStart st) {
  const int lane = threadIdx.x & 31;
  Ring R{st.issued % M.S, st.issued / M.S, M.S};
  // A stage is refilled once the consumers released it and its previous fill
  // has landed -- immediate unless a timeout let the consumers skip their
  // wait: one fill per barrier phase.
  auto take_stage = [&]() -> uint8_t* {
    if (R.use > 0) {
      if (lane == 0) {
        mbar_wait_bounded(&E.empty[R.slot], (R.use - 1) & 1, &E.wc, C.status);
        mbar_drain(&E.full[R.slot], (R.use - 1) & 1);
      }
      __syncwarp();
    }
    return M.stages + (size_t)R.slot * M.SB;
  };
  int cur = st.j, first = st.issued;
  for (int pos = 0, n = 1;; ++pos, ++n) {
    UnitInfo u;
    const bool more = sch.unit(cur, u);
    if (!more) u.kind = kItemEnd;
    if (lane == 0) ring_put(E, pos, u, C.status);
    __syncwarp();
    if (!more) break;
    int nxt = 0;
    if (lane == 0) nxt = sch.claim(n);
    if (u.kind != kItemCombine) {
      const MatGeo& g = C.geo[u.mat];
      for (int c = first; c < u.nch; ++c) {
        produce_weights(g, u, c, take_stage(), &E.full[R.slot]);
        R.next();
        if (pos == 0 && c == 0) {  // the call's first copy lands first
          if (lane == 0) mbar_wait_bounded(&E.full[0], 0, &E.wc, C.status);
          __syncwarp();
        }
      }
    }
    first = 0;
    cur = __shfl_sync(0xffffffffu, nxt, 0);
    if (lane == 0) {
      UnitInfo t;
      if (sch.unit(cur, t)) prefetch_unit(C, t, 0);
    }
  }
  // wait until the last copies have landed (every stage's most recent fill),
  // also after a timeout: the CTA may not exit with copies into its shared
  // memory in flight
  if (lane == 0)
    for (int s = 0; s < M.S; ++s) {
      const int uses = R.use + (s < R.slot ? 1 : 0);
      if (uses > 0) mbar_drain(&E.full[s], (uses - 1) & 1);
    }
  __syncwarp();
}

// The operand warp's loop: per unit, an operand buffer once the consumers
// released it (and its previous fill landed), after the unit's dependency
// on other CTAs.  A combine piece gets an empty fill that only signals that
// its y rows are complete.
template <class Sched>
__device__ void operand_run(const EngineCfg& C, EngineSmem& E, const EngineMem& M,
                            const Sched& sch, const int* ctrl) {
  const int lane = threadIdx.x & 31;
  Ring B{0, 0, M.nob};
  for (int pos = 0;; ++pos) {
    const UnitInfo u = ring_take(E, pos, C.status);
    if (u.kind == kItemEnd) break;
    if (B.use > 0) {
      if (lane == 0) {
        mbar_wait_bounded(&E.op_empty[B.slot], (B.use - 1) & 1, &E.wc, C.status);
        mbar_drain(&E.op_full[B.slot], (B.use - 1) & 1);
      }
      __syncwarp();
    }
    if (u.kind == kItemCombine) {
      if (lane == 0) {
        wait_counter(ctrl + u.wait_ctr, u.wait_target, &E.wc, C.status);
        mbar_arrive(&E.op_full[B.slot]);
      }
      __syncwarp();
    } else {
      produce_operands(C, sch.source(u.mat), u, sch.perm(), sch.topk(),
                       M.ops + (size_t)B.slot * M.OB, &E.op_full[B.slot], ctrl, &E.wc);
    }
    B.next();
  }
  if (lane == 0)
    for (int b = 0; b < M.nob; ++b) {
      const int uses = B.use + (b < B.slot ? 1 : 0);
      if (uses > 0) mbar_drain(&E.op_full[b], (uses - 1) & 1);
    }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Consumer epilogues (all 512 consumer threads).

// SwiGLU of a gate/up unit: warps with tile < 4 hold gate rows 64 blk + 16
// tile + {g, g+8}, tiles 4..7 the matching up rows; the k-groups are added
// first, in order.
//   h = a / (1 + exp(-a)) * u,  hi = bf16(h), lo = bf16(h - hi)
// stored at output row out_row(n), columns 64 blk + r, and the padded sum
// over the 64 rows of (hi + lo) in a fixed tree (32 rows by shuffles, then
// the two warps of the token in order).
__device__ __forceinline__ void epilogue_gateup(const EngineCfg& C, EngineSmem& E,
                                                const UnitInfo& u, int my_orow,
                                                const float (&acc)[4]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = warp % kTiles, ks = warp / kTiles;
#pragma unroll
  for (int i = 0; i < 4; ++i) E.red[ks][tile][lane][i] = acc[i];
  consumer_sync();
  const MatTarget& T = C.tg[u.mat];
  const int I = C.inter;
  const int n = warp >> 1, r = (warp & 1) * 32 + lane;
  const int tl = r >> 4, rr = r & 15;
  const int src = (rr & 7) * 4 + (n >> 1), idx = (rr >> 3) * 2 + (n & 1);
  const float a = E.red[0][tl][src][idx] + E.red[1][tl][src][idx];
  const float up = E.red[0][tl + 4][src][idx] + E.red[1][tl + 4][src][idx];
  const float h = a / (1.f + expf(-a)) * up;
  const __nv_bfloat16 hb = __float2bfloat16_rn(h);
  const __nv_bfloat16 lb = __float2bfloat16_rn(h - __bfloat162float(hb));
  float s = __bfloat162float(hb) + __bfloat162float(lb);
  const int o = __shfl_sync(0xffffffffu, my_orow, n);
  if (n < u.cnt) {
    const size_t at = (size_t)o * h_pitch(I) + u.blk * 64 + r;
    T.hh[at] = __bfloat16_as_ushort(hb);
    T.hl[at] = __bfloat16_as_ushort(lb);
    if (T.hout) T.hout[(size_t)o * I + u.blk * 64 + r] = h;
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
  if (lane == 0) E.part[warp] = s;
  consumer_sync();
  if (warp == 0) {
    const TileGeo& dg = C.geo[u.mat | 1].t;  // the down matrix reads these sums
    const int o2 = __shfl_sync(0xffffffffu, my_orow, lane & 7);
    if (lane < u.cnt)
      T.hsum[(size_t)o2 * sums_ld(dg) + sums_pos(dg, u.blk)] =
          E.part[2 * lane] + E.part[2 * lane + 1];
  }
}

// Output of a down unit: each warp writes its k-half's sums straight to its
// plane of y (plane kh, row out_row(n), column 128 blk + 16 tile + g (+8));
// the two planes are added (plane 0 + plane 1) where y is read.
__device__ __forceinline__ void epilogue_down(const EngineCfg& C, const UnitInfo& u,
                                              int my_orow, const float (&acc)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tile = warp & 7, kh = warp >> 3;
  const int g = lane >> 2, t = lane & 3;
  const MatTarget& T = C.tg[u.mat];
  float* y = T.y + (kh ? T.yhalf : 0) + u.blk * kUnitRows + tile * 16 + g;
  const int H = C.hidden;
  const int o0 = __shfl_sync(0xffffffffu, my_orow, (2 * t) & 7);
  const int o1 = __shfl_sync(0xffffffffu, my_orow, (2 * t + 1) & 7);
  if (2 * t < u.cnt) {
    y[(size_t)o0 * H] = acc[0];
    y[(size_t)o0 * H + 8] = acc[2];
  }
  if (2 * t + 1 < u.cnt) {
    y[(size_t)o1 * H] = acc[1];
    y[(size_t)o1 * H + 8] = acc[3];
  }
}

// ---------------------------------------------------------------------------
// Publishing finished units.  After a unit's results are written, every
// consumer warp arrives on epi_full[slot]; the signal warp waits for it and
// adds 1 to the unit's control word with a release reduction (cumulative: it
// publishes every write the signal warp has observed through the barrier),
// then frees the slot.  Units without a control word skip all of this.
__device__ __forceinline__ void epi_publish(EngineSmem& E, Ring& P, const UnitInfo& u,
                                            int* status) {
  if (u.signal < 0) return;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    if (P.use > 0) mbar_wait_bounded(&E.epi_empty[P.slot], (P.use - 1) & 1, &E.wc, status);
    mbar_arrive(&E.epi_full[P.slot]);
  }
  P.next();
}

template <class Sched>
__device__ void signal_run(EngineSmem& E, const Sched& sch, int* ctrl, int* status) {
  const int lane = threadIdx.x & 31;
  Ring P{0, 0, kEpiRing};
  (void)sch;
  for (int pos = 0;; ++pos) {
    const UnitInfo u = ring_take(E, pos, status);
    if (u.kind == kItemEnd) break;
    if (u.kind == kItemCombine || u.signal < 0) continue;
    if (lane == 0) {
      mbar_wait_bounded(&E.epi_full[P.slot], P.use & 1, &E.wc, status);
      red_release_add(ctrl + u.signal, 1);
      mbar_arrive(&E.epi_empty[P.slot]);
    }
    __syncwarp();
    P.next();
  }
}

// ---------------------------------------------------------------------------
// Consumers' loop over the units of the ring.  sch.combine(blk) runs a
// combine piece (fused kernel only).
template <int FMT, int FMT_SH, bool F16A, class Sched>
__device__ void consumer_run(const EngineCfg& C, EngineSmem& E, const EngineMem& M,
                             const Sched& sch) {
  const int lane = threadIdx.x & 31;
  Ring R{0, 0, M.S}, B{0, 0, M.nob}, P{0, 0, kEpiRing};
  float acc[4];
  for (int pos = 0;; ++pos) {
    const UnitInfo u = ring_take(E, pos, C.status);
    if (u.kind == kItemEnd) break;
    if (u.kind == kItemCombine) {
      mbar_wait_bounded(&E.op_full[B.slot], B.use & 1, &E.wc, C.status);
      sch.combine(u.blk);
      __syncwarp();
      if (lane == 0) mbar_arrive(&E.op_empty[B.slot]);
      B.next();
      continue;
    }
    const int my_orow = lane < u.cnt ? unit_out_row(u, sch.perm(), lane) : 0;
    const uint8_t* op = M.ops + (size_t)B.slot * M.OB;
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    unit_mat<FMT, FMT_SH, F16A>(C, u.mat, E, M, R, op, &E.op_full[B.slot], B.use & 1, acc);
    if (lane == 0) mbar_arrive(&E.op_empty[B.slot]);
    B.next();
    if (u.kind == kItemDown)
      epilogue_down(C, u, my_orow, acc);
    else
      epilogue_gateup(C, E, u, my_orow, acc);
    epi_publish(E, P, u, C.status);
  }
}

// ---------------------------------------------------------------------------
// Weighted combine of output columns [h0, h0 + nh), for all T tokens:
//   out[t, h] = round( sum_j w[t, j] * y[t*k + j, h]  +  s_t * ysh[t, h] )
// an fp32 fma chain in slot order with the shared slot last; y comes as two
// k-half planes added plane 0 + plane 1 first (one plane when yhalf == 0),
// ysh likewise when ysh2 is given.  rb rounds the weights w and sg to bf16
// first (the engine's bf16 rounding chain; idempotent on rounded weights).
// y and ysh are read through L2 (written by other CTAs); every load of one
// output is issued before the chain starts (k <= kMaxTopK).  `nthr` threads.
constexpr int kMaxTopK = 8;
constexpr int kCombineRows = 64;  // columns of one combine piece
// In the prefill form (one_plane set) an assignment whose expert has more
// than one_plane_max assignments (by the bucket offsets) has its y in plane 0
// alone (the tensor-core GEMMs); the second plane is then taken as 0.
__device__ __forceinline__ void combine_rows(const float* y, size_t yhalf, const float* w,
                                             const float* ysh, const float* ysh2,
                                             const float* sg, uint16_t* out, int T, int k, int H,
                                             bool f16, int h0, int nh, int tid, int nthr,
                                             bool rb = false, const int32_t* idx = nullptr,
                                             const int32_t* offsets = nullptr,
                                             int one_plane_max = 0) {
  for (int v = tid; v < T * nh; v += nthr) {
    const int t = v / nh;
    const int h = h0 + (v - t * nh);
    float ya[kMaxTopK], yb[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {
        const size_t a = (size_t)(t * k + j) * H + h;
        ya[j] = __ldcg(y + a);
        bool two = yhalf != 0;
        if (two && idx) {
          const int e = __ldg(idx + t * k + j);
          two = __ldg(offsets + e + 1) - __ldg(offsets + e) <= one_plane_max;
        }
        yb[j] = two ? __ldcg(y + yhalf + a) : 0.f;
      }
    }
    float vs = 0.f;
    if (ysh) {
      const size_t a = (size_t)t * H + h;
      vs = ysh2 ? __ldcg(ysh + a) + __ldcg(ysh2 + a) : __ldcg(ysh + a);
    }
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) {
        const float wj = rb ? round_bf16(w[t * k + j]) : w[t * k + j];
        acc = fmaf(wj, yhalf ? ya[j] + yb[j] : ya[j], acc);
      }
    if (ysh) acc = fmaf(sg ? (rb ? round_bf16(sg[t]) : sg[t]) : 1.f, vs, acc);
    out[(size_t)t * H + h] = float_to_act_bits(acc, f16);
  }
}

// Per-64-group sums of activation rows, in the padded layout: one warp per
// (token, 128 columns); lane l adds its 4 values in order, then 16 lanes in a
// fixed xor tree.  `task` enumerates (t, 128-column block).
__device__ __forceinline__ void xsum_task(const uint16_t* x, int H, bool f16, const TileGeo& g13,
                                          float* xsum, int task) {
  const int lane = threadIdx.x & 31;
  const int nb = H >> 7;
  const int t = task / nb, q = task - t * nb;
  const uint2 v = *reinterpret_cast<const uint2*>(x + (size_t)t * H + q * 128 + 4 * lane);
  float s = act_to_float(uint16_t(v.x & 0xFFFFu), f16);
  s += act_to_float(uint16_t(v.x >> 16), f16);
  s += act_to_float(uint16_t(v.y & 0xFFFFu), f16);
  s += act_to_float(uint16_t(v.y >> 16), f16);
#pragma unroll
  for (int m = 8; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
  if ((lane & 15) == 0) {
    const int j = 2 * q + (lane >> 4);
    xsum[(size_t)t * sums_ld(g13) + sums_pos(g13, j)] = s;
  }
}

}  // namespace moe
