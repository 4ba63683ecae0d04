// engine.cuh -- the warp-specialised item engine of the decode path, shared
// by the standalone expert kernels (units.cu) and the fused layer kernel
// (decode.cu).
//
// A CTA has 17 warps: warp 16 is the producer, warps 0..15 the consumers.
// Work comes as "units": one sub-slot (<= 8 tokens of one expert) times one
// 128-row block of a matrix, streamed as k-chunk "items".  An item is a
// contiguous block of the kernel-tiled bank (codes + scales, tiled.cuh) plus
// the operand rows (x, or h as bf16 hi + lo) and their per-64-group sums.
//   producer: for each item, waits until its stage is free (empty barrier),
//             writes a small descriptor into the stage, and fills the stage
//             with TMA bulk copies that complete on the stage's full barrier;
//             it alone waits on other CTAs (operands produced in the kernel).
//   consumers: wait for the full barrier, run the MMA pass over the item,
//             release the stage, and after the last item of a unit reduce and
//             write the unit's result (SwiGLU -> h, or y).
// There is no CTA-wide barrier in the item loop; consumers synchronise only
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
// call or on its sub-slot, and the fused and standalone kernels (same device
// functions) give the same bits.
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
constexpr int kEngineThreads = kConsumers + 32;     // + the producer warp
constexpr int kProducerWarp = kConsumerWarps;
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

// Item descriptor, written by the producer at the start of the stage.
enum : int { kItemGateUp = 0, kItemDown = 1, kItemCombine = 2, kItemEnd = 3 };

struct ItemDesc {
  int kind;
  int mat;     // 0 routed w13, 1 routed w2, 2 shared w13, 3 shared w2
  int c;       // k-chunk
  int first;   // first chunk of its unit (clear the accumulators)
  int last;    // last chunk (epilogue)
  int cnt;     // tokens, 1..8
  int blk;     // 64-row group (gate/up), 128-row block (down, combine)
  int signal;  // control word to add 1 to after the epilogue, -1 for none
  int orow[kMaxTok];  // output row of token slot n (h row, or y row)
};

// Shared-memory stage: [descriptor][tiled item][operand hi][operand lo][sums]
struct StageLayout {
  int a, x, xlo, xs, bpitch, ngp, bytes;
};

__host__ __device__ inline StageLayout stage_layout(const TileGeo& t) {
  StageLayout L;
  L.bpitch = t.CK * 2 + 16;  // operand rows 16 bytes past a multiple of 128
  L.ngp = sums_ngp(t);
  L.a = 128;
  L.x = L.a + align128i(t.item_bytes);
  L.xlo = L.x + kMaxTok * L.bpitch;
  L.xs = t.down ? L.xlo + kMaxTok * L.bpitch : L.xlo;
  L.bytes = align128i(L.xs + kMaxTok * L.ngp * 4);
  return L;
}

// Bytes a stage receives for an item of `cnt` tokens.
__host__ __device__ inline unsigned item_tx_bytes(const TileGeo& t, int cnt) {
  const int rowb = t.CK * 2 * (t.down ? 2 : 1) + sums_ngp(t) * 4;
  return unsigned(t.item_bytes + cnt * rowb);
}

// Where the consumers' results go, per matrix slot.
struct MatTarget {
  uint16_t* hh;   // gate/up: h hi part [rows][I] (bf16)
  uint16_t* hl;   //          h lo part
  float* hsum;    //          padded sums of hi + lo per 64-group
  float* hout;    //          nullable fp32 h
  float* y;       // down:    [rows][H] fp32
};

struct EngineCfg {
  MatGeo geo[4];
  MatTarget tg[4];
  int fmt_shared;  // format of the shared bank (slots 2, 3)
  int inter, hidden;
  int* status;     // device status word
};

// ---------------------------------------------------------------------------
// Barrier helpers (all waits bounded).

// Wait for phase `parity` of an mbarrier; on the limit, record a timeout and
// return false.  `skip` (shared) turns every later wait into a no-op once a
// timeout has happened, so the kernel finishes (with garbage results) quickly.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity,
                                                  volatile int* skip, int* status) {
  for (int i = 0; i < (1 << 22); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && *skip) return false;
  }
  *skip = 1;
  atomicExch(status, int(MOE_ERR_TIMEOUT));
  return false;
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

__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait (one thread) until *p >= target; on the limit records a timeout
// and sets *skip.  Returns at once when *skip is already set.
static __device__ __noinline__ bool wait_counter(const int* p, int target, volatile int* skip,
                                          int* status) {
  unsigned ns = 32;
  for (int i = 0; i < (1 << 21); ++i) {
    if (ld_acquire(p) >= target) return true;
    if (*skip) return false;
    __nanosleep(ns);
    if (ns < 256) ns <<= 1;
  }
  *skip = 1;
  atomicExch(status, int(MOE_ERR_TIMEOUT));
  return false;
}

}  // namespace moe

namespace moe {

// ---------------------------------------------------------------------------
// Consumer arithmetic.

// Two codes (bits [0,4) and [16,20) of v) -> two 16-bit floats.  bf16: the
// code is ORed into the mantissa of 128.0 (0x4300), giving exactly 128 + q;
// the 128 is taken out in the fold (bias' = bias - 128 scale).  fp16: 1024 + q
// (0x6400) minus 1024, exact, so the operand is q itself.
template <bool F16>
__device__ __forceinline__ uint32_t code_pair(uint32_t v) {
  if constexpr (F16) {
    uint32_t r = (v & 0x000F000Fu) | 0x64006400u;
    __half2 h = *reinterpret_cast<__half2*>(&r);
    const __half2 off = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    h = __hsub2(h, off);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    return (v & 0x000F000Fu) | 0x43004300u;
  }
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t v) {
  return __half22float2(*reinterpret_cast<__half2*>(&v));
}

// One k-chunk item for consumer warp (tile, kh): groups [kh*ng/2, (kh+1)*ng/2)
// of M-tile `tile`, added into acc.  acc[0]: (row g, token 2t), acc[1]:
// (g, 2t+1), acc[2]: (g+8, 2t), acc[3]: (g+8, 2t+1).  Operand columns of
// tokens >= cnt hold whatever the stage held before; MMA columns are
// independent, so they only touch accumulators that are never written out.
template <int FMT, bool F16A, bool SPLIT>
__device__ __forceinline__ void compute_item(const TileGeo& tg, const uint8_t* st,
                                             const StageLayout& L, int tile, int kh,
                                             float (&acc)[4]) {
  constexpr int CB = FMT == MOE_FMT_AFFINE3_G64 ? 384 : 512;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;
  const int ng = tg.ng, gh = ng >> 1, G0 = kh * gh;
  const uint8_t* codes = st + L.a + (tile * ng + G0) * CB;
  const uint8_t* xrow = st + L.x + gq * L.bpitch + G0 * 128 + 32 * t;
  const uint8_t* xlrow = st + L.xlo + gq * L.bpitch + G0 * 128 + 32 * t;
  const float* xs0 = reinterpret_cast<const float*>(st + L.xs) + (2 * t) * L.ngp + G0;
  const float* xs1 = xs0 + L.ngp;
  const uint8_t* sc = st + L.a + tg.code_bytes;
#pragma unroll 2
  for (int G = 0; G < gh; ++G) {
    uint32_t w0, w1, w2, w3;
    if constexpr (FMT == MOE_FMT_AFFINE3_G64) {
      const uint32_t* pl = reinterpret_cast<const uint32_t*>(codes + G * 384) + lane;
      planes_to_words(pl[0], pl[32], pl[64], w0, w1, w2, w3);
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(codes + G * 512 + lane * 16);
      w0 = v.x;
      w1 = v.y;
      w2 = v.z;
      w3 = v.w;
    }
    const uint4 xa = *reinterpret_cast<const uint4*>(xrow + G * 128);
    const uint4 xb = *reinterpret_cast<const uint4*>(xrow + G * 128 + 16);
    // k-step m takes code pairs (4m, 4m+1) and (4m+2, 4m+3) of the lane's 16
    // codes: nibbles (m&1)*2 and (m&1)*2+1 of word W0/W1 (row g), W2/W3 (g+8)
    const uint32_t A00 = code_pair<F16A>(w0), A01 = code_pair<F16A>(w2);
    const uint32_t A02 = code_pair<F16A>(w0 >> 4), A03 = code_pair<F16A>(w2 >> 4);
    const uint32_t A10 = code_pair<F16A>(w0 >> 8), A11 = code_pair<F16A>(w2 >> 8);
    const uint32_t A12 = code_pair<F16A>(w0 >> 12), A13 = code_pair<F16A>(w2 >> 12);
    const uint32_t A20 = code_pair<F16A>(w1), A21 = code_pair<F16A>(w3);
    const uint32_t A22 = code_pair<F16A>(w1 >> 4), A23 = code_pair<F16A>(w3 >> 4);
    const uint32_t A30 = code_pair<F16A>(w1 >> 8), A31 = code_pair<F16A>(w3 >> 8);
    const uint32_t A32 = code_pair<F16A>(w1 >> 12), A33 = code_pair<F16A>(w3 >> 12);
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
    float s0, s1, b0, b1;
    if constexpr (FMT == MOE_FMT_W4A16_SYM_G128) {
      const uint32_t sv = *reinterpret_cast<const uint32_t*>(
          sc + ((tile * 8 + gq) * (ng >> 1) + ((G0 + G) >> 1)) * 4);
      const float2 sf = half2_bits_to_float2(sv);
      s0 = sf.x;
      s1 = sf.y;
      // w = s (u - 8) for the stored nibble u; with the bf16 operand's +128
      // the offset is -136 s (exact: an fp16 times 136 fits in fp32)
      b0 = (F16A ? -8.f : -136.f) * s0;
      b1 = (F16A ? -8.f : -136.f) * s1;
    } else {
      const uint2 sv =
          *reinterpret_cast<const uint2*>(sc + ((tile * 8 + gq) * ng + G0 + G) * 8);
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

// Format dispatch of one item (mat: 0/2 gate/up, 1/3 down).
template <int FMT, bool F16A>
__device__ __forceinline__ void compute_mat(const EngineCfg& C, int mat, const uint8_t* st,
                                            int tile, int kh, float (&acc)[4]) {
  const TileGeo& tg = C.geo[mat].t;
  const StageLayout L = stage_layout(tg);
  const bool down = mat & 1;
  if (mat < 2) {
    if (down)
      compute_item<FMT, false, true>(tg, st, L, tile, kh, acc);
    else
      compute_item<FMT, F16A, false>(tg, st, L, tile, kh, acc);
    return;
  }
  switch (C.fmt_shared) {
    case MOE_FMT_AFFINE3_G64:
      if (down)
        compute_item<MOE_FMT_AFFINE3_G64, false, true>(tg, st, L, tile, kh, acc);
      else
        compute_item<MOE_FMT_AFFINE3_G64, F16A, false>(tg, st, L, tile, kh, acc);
      break;
    case MOE_FMT_W4A16_SYM_G128:
      if (down)
        compute_item<MOE_FMT_W4A16_SYM_G128, false, true>(tg, st, L, tile, kh, acc);
      else
        compute_item<MOE_FMT_W4A16_SYM_G128, F16A, false>(tg, st, L, tile, kh, acc);
      break;
    default:
      if (down)
        compute_item<MOE_FMT_AFFINE4_G64, false, true>(tg, st, L, tile, kh, acc);
      else
        compute_item<MOE_FMT_AFFINE4_G64, F16A, false>(tg, st, L, tile, kh, acc);
      break;
  }
}

}  // namespace moe

namespace moe {

// ---------------------------------------------------------------------------
// Units and where their rows come from / go to.

// Operand source of a matrix slot: rows of B (and Blo) of ldB elements, and
// their padded per-64-group sums (row stride ldS floats).
struct MatSource {
  const uint16_t* B;
  const uint16_t* Blo;  // nullptr unless the operand is split (h)
  const float* Bsum;
  int ldB, ldS;
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
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int skip;                       // set after the first timeout
  float red[2][8][32][4];         // epilogue: accumulators by k-half, tile, lane
  float part[kConsumerWarps];     // epilogue: per-warp partial sums
};

__device__ __forceinline__ void engine_init(EngineSmem& E, int S) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&E.full[s], 1);
      mbar_init(&E.empty[s], kConsumerWarps);
    }
    E.skip = 0;
  }
}

// Stage ring position: slot and how many times it has been used.
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
// Producer (warp kProducerWarp, all 32 lanes).

// Fill stage `st` with item (u, c): the tiled item by four bulk copies, then
// (after the unit's dependency, for the first chunk) the operand rows and
// their sums, one bulk copy per row.  Completes on *full.
__device__ __forceinline__ void produce_item(const EngineCfg& C, const MatSource& src,
                                             const UnitInfo& u, int c, const int* perm, int k,
                                             uint8_t* st, uint64_t* full, const int* ctrl,
                                             volatile int* skip) {
  const int lane = threadIdx.x & 31;
  const TileGeo& tg = C.geo[u.mat].t;
  const StageLayout L = stage_layout(tg);
  if (lane == 0) mbar_expect_only(full, item_tx_bytes(tg, u.cnt));
  __syncwarp();
  const int bytes = tg.item_bytes;
  if (lane < 4) {
    const uint8_t* w = C.geo[u.mat].base + (size_t)u.e * tg.expert_bytes +
                       (size_t)(u.blk * tg.nch + c) * bytes;
    const int piece = align16i((bytes + 3) / 4);
    const int o = lane * piece;
    const int n = min(piece, bytes - o);
    if (n > 0) bulk_g2s(st + L.a + o, w + o, unsigned(n), full);
  }
  if (u.wait_ctr >= 0 && c == 0) {
    if (lane == 0) wait_counter(ctrl + u.wait_ctr, u.wait_target, skip, C.status);
    __syncwarp();
    fence_proxy_async_global();
  }
  // lanes 8..15: operand hi rows, 16..23: lo rows, 24..31: sums
  const int part = lane >> 3, n = lane & 7;
  if (part >= 1 && n < u.cnt) {
    const int row = unit_op_row(u, perm, k, n);
    if (part == 1) {
      bulk_g2s(st + L.x + n * L.bpitch, src.B + (size_t)row * src.ldB + (size_t)c * tg.CK,
               unsigned(tg.CK * 2), full);
    } else if (part == 2) {
      if (src.Blo)
        bulk_g2s(st + L.xlo + n * L.bpitch, src.Blo + (size_t)row * src.ldB + (size_t)c * tg.CK,
                 unsigned(tg.CK * 2), full);
    } else {
      bulk_g2s(st + L.xs + n * L.ngp * 4, src.Bsum + (size_t)row * src.ldS + (size_t)c * L.ngp,
               unsigned(L.ngp * 4), full);
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(full);
}

// The producer's loop over a schedule (sch.n_units(), sch.unit(j)).
template <class Sched>
__device__ void producer_run(const EngineCfg& C, EngineSmem& E, uint8_t* stages, int SB, int S,
                             const Sched& sch, const int* ctrl) {
  const int lane = threadIdx.x & 31;
  Ring R{0, 0, S};
  int issued = 0;
  const int nu = sch.n_units();
  for (int j = 0; j < nu; ++j) {
    const UnitInfo u = sch.unit(j);
    const int nit = u.kind == kItemCombine ? 1 : u.nch;
    for (int c = 0; c < nit; ++c) {
      if (R.use > 0) {
        if (lane == 0) mbar_wait_bounded(&E.empty[R.slot], (R.use - 1) & 1, &E.skip, C.status);
        __syncwarp();
      }
      uint8_t* st = stages + (size_t)R.slot * SB;
      if (u.kind == kItemCombine) {
        if (lane == 0) {
          wait_counter(ctrl + u.wait_ctr, u.wait_target, &E.skip, C.status);
          mbar_arrive(&E.full[R.slot]);
        }
        __syncwarp();
      } else {
        produce_item(C, sch.source(u.mat), u, c, sch.perm(), sch.topk(), st, &E.full[R.slot],
                     ctrl, &E.skip);
      }
      ++issued;
      R.next();
    }
  }
  // wait (bounded) until every stage this warp filled has landed
  if (lane == 0) {
    Ring D{0, 0, S};
    for (int i = 0; i < issued; ++i) {
      if (i + S >= issued) mbar_wait_bounded(&E.full[D.slot], D.use & 1, &E.skip, C.status);
      D.next();
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Consumer epilogues (all 512 consumer threads).

// SwiGLU of a gate/up unit: warps with tile < 4 hold gate rows 64 blk + 16
// tile + {g, g+8}, tiles 4..7 the matching up rows; k-halves are added first.
//   h = a / (1 + exp(-a)) * u,  hi = bf16(h), lo = bf16(h - hi)
// stored at output row out_row(n), columns 64 blk + r, and the padded sum
// over the 64 rows of (hi + lo) in a fixed tree (32 rows by shuffles, then
// the two warps of the token in order).
__device__ __forceinline__ void epilogue_gateup(const EngineCfg& C, EngineSmem& E,
                                                const UnitInfo& u, int my_orow,
                                                const float (&acc)[4], int* ctrl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = warp & 7, kh = warp >> 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) E.red[kh][tile][lane][i] = acc[i];
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
    const size_t at = (size_t)o * I + u.blk * 64 + r;
    T.hh[at] = __bfloat16_as_ushort(hb);
    T.hl[at] = __bfloat16_as_ushort(lb);
    if (T.hout) T.hout[at] = h;
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
    __syncwarp();
    if (lane == 0 && u.signal >= 0) {
      __threadfence();
      red_release_add(ctrl + u.signal, 1);
    }
  }
}

// Output of a down unit: y[out_row(n)][128 blk + r] = k-half 0 + k-half 1.
__device__ __forceinline__ void epilogue_down(const EngineCfg& C, EngineSmem& E,
                                              const UnitInfo& u, int my_orow,
                                              const float (&acc)[4], int* ctrl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = warp & 7, kh = warp >> 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) E.red[kh][tile][lane][i] = acc[i];
  consumer_sync();
  float* y = C.tg[u.mat].y;
  const int H = C.hidden;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int v = tid + kConsumers * s;
    const int n = v >> 7, r = v & 127;
    const int tl = r >> 4, rr = r & 15;
    const int src = (rr & 7) * 4 + (n >> 1), idx = (rr >> 3) * 2 + (n & 1);
    const int o = __shfl_sync(0xffffffffu, my_orow, n);
    if (n < u.cnt)
      y[(size_t)o * H + u.blk * kUnitRows + r] = E.red[0][tl][src][idx] + E.red[1][tl][src][idx];
  }
  consumer_sync();
  if (tid == 0 && u.signal >= 0) {
    __threadfence();
    red_release_add(ctrl + u.signal, 1);
  }
}

// ---------------------------------------------------------------------------
// Consumers' loop over the same schedule as the producer.  sch.combine(blk)
// runs a combine unit (fused kernel only).
template <int FMT, bool F16A, class Sched>
__device__ void consumer_run(const EngineCfg& C, EngineSmem& E, const uint8_t* stages, int SB,
                             int S, const Sched& sch, int* ctrl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tile = warp & 7, kh = warp >> 3;
  Ring R{0, 0, S};
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int nu = sch.n_units();
  for (int j = 0; j < nu; ++j) {
    const UnitInfo u = sch.unit(j);
    if (u.kind == kItemCombine) {
      mbar_wait_bounded(&E.full[R.slot], R.use & 1, &E.skip, C.status);
      __syncwarp();
      if (lane == 0) mbar_arrive(&E.empty[R.slot]);
      R.next();
      sch.combine(u.blk);
      continue;
    }
    const int my_orow = lane < u.cnt ? unit_out_row(u, sch.perm(), lane) : 0;
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    for (int c = 0; c < u.nch; ++c) {
      mbar_wait_bounded(&E.full[R.slot], R.use & 1, &E.skip, C.status);
      compute_mat<FMT, F16A>(C, u.mat, stages + (size_t)R.slot * SB, tile, kh, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&E.empty[R.slot]);
      R.next();
    }
    if (u.kind == kItemDown)
      epilogue_down(C, E, u, my_orow, acc, ctrl);
    else
      epilogue_gateup(C, E, u, my_orow, acc, ctrl);
  }
}

// ---------------------------------------------------------------------------
// Weighted combine of one 128-row block of the output, for all T tokens:
//   out[t, h] = round( sum_j w[t, j] * y[t*k + j, h]  +  s_t * ysh[t, h] )
// an fp32 fma chain in slot order with the shared slot last.  y and ysh are
// read through L2 (written by other CTAs).  `nthr` threads from `tid0`.
__device__ __forceinline__ void combine_rows(const float* y, const float* w, const float* ysh,
                                             const float* sg, uint16_t* out, int T, int k, int H,
                                             bool f16, int blk, int tid, int nthr) {
  for (int v = tid; v < T * kUnitRows; v += nthr) {
    const int t = v >> 7;
    const int h = blk * kUnitRows + (v & 127);
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
      const int a = t * k + j;
      acc = fmaf(w[a], __ldcg(y + (size_t)a * H + h), acc);
    }
    if (ysh) acc = fmaf(sg ? sg[t] : 1.f, __ldcg(ysh + (size_t)t * H + h), acc);
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
