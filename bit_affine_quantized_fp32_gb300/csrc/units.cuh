// units.cuh -- the decode-path work unit shared by the standalone expert
// kernels and the fused persistent layer kernel.
//
// Tokens of one expert are cut into sub-slots of at most 8 (one MMA n-tile).
// A unit is one CTA (8 warps) x one sub-slot x 128 weight rows:
//   gate/up unit: gate rows [64j, 64j+64) and up rows [I+64j, I+64j+64) of w13
//                 over the whole hidden dimension, so its epilogue applies
//                 SwiGLU and writes h for that 64-row group directly;
//   down unit:    rows [128r, 128r+128) of w2 over the whole intermediate.
// A unit is streamed as k-chunks ("items"); warp w owns the 16-row M-tile w
// and keeps its fp32 accumulators in registers across the items.  The codes,
// fp16 scales/biases and the operand rows of an item are staged in shared
// memory by 16-byte cp.async; three stages keep two items in flight.
//
// Arithmetic per weight row r, 64-code group G and token n:
//   sum_i (s q_i + b) x_i = s * (sum_i q_i x_i) + b * X_G(n)
// The bracket is an mma.sync m16n8k16 with the codes as exact bf16/fp16
// integers (fp32 accumulation, exact products); s and b are applied in fp32.
// The down operand h (fp32) goes through as two bf16 parts hi + lo.
//
// Fragment mapping (see also kperm_pos): thread (g = lane/4, t = lane%4) takes
// packed words 2t and 2t+1 of rows g and g+8 of the group (codes 16t..16t+15);
// nibble pairs (0,4) (1,5) (2,6) (3,7) of a word are the MMA k-pairs, and the
// operand rows are stored with each 8-block permuted to [0 4 1 5 2 6 3 7].
//
// Every output element is one MMA column with a fixed k-order (chunks, groups,
// MMA steps) and fixed fp32 folds and reductions, so a token's result never
// depends on the other tokens of the call or on its sub-slot.
#pragma once

#include "common.cuh"
#include "tiled.cuh"

namespace moe {

constexpr int kUnitThreads = 256;
constexpr int kUnitWarps = 8;
constexpr int kUnitRows = 128;
constexpr int kMaxTok = 8;
constexpr int kStages = 3;

__host__ __device__ inline int align16i(int x) { return (x + 15) & ~15; }

// A matrix family (w13 or w2) of a tiled bank.
struct MatGeo {
  TileGeo t;
  const uint8_t* base;   // tiled buffer (expert 0, item 0)
};

// Shared-memory stage: [tiled item (codes + scales)][operand rows hi][lo][sums]
struct StageLayout {
  int a, x, xlo, xsum, bpitch, bytes;
};

__host__ __device__ inline StageLayout stage_layout(const TileGeo& t) {
  StageLayout L;
  L.bpitch = t.CK * 2 + 16;  // operand rows 16 bytes past a multiple of 128
  int o = 0;
  L.a = o;
  o += align16i(t.item_bytes);
  L.x = o;
  o += kMaxTok * L.bpitch;
  L.xlo = o;
  o += kMaxTok * L.bpitch;
  L.xsum = o;
  o += align16i(kMaxTok * t.ng * 4);
  L.bytes = o;
  return L;
}

// One resolved unit.
struct Unit {
  int down;   // 0: gate/up unit, 1: down unit
  int e;      // expert
  int blk;    // 64-row group of the intermediate (gate/up) or 128-row block (down)
  int off;    // first bucket position (or token) of the sub-slot
  int cnt;    // tokens of the sub-slot, 1..8
  int ss;     // sub-slot index
};

// Stage the tiled item (unit, chunk c) by TMA bulk copies issued from warp 0
// (four pieces of ~9 KiB), completing on `bar` with the item's byte count.
__device__ __forceinline__ void stage_weights(const MatGeo& g, const Unit& u, int c, uint8_t* st,
                                              const StageLayout& L, uint64_t* bar) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int bytes = g.t.item_bytes;
  const uint8_t* src = g.base + (size_t)u.e * g.t.expert_bytes +
                       (size_t)(u.blk * g.t.nch + c) * bytes;
  const int piece = align16i((bytes + 3) / 4);
  if (lane == 0) mbar_expect_tx(bar, unsigned(bytes));
  __syncwarp();
  if (lane < 4) {
    const int o = lane * piece;
    const int n = min(piece, bytes - o);
    if (n > 0) bulk_g2s(st + L.a + o, src + o, unsigned(n), bar);
  }
}

// Row of token n < ntok in the operand: rowmap[base + n] (or base + n without
// a map; rowmap may point to shared memory).
__device__ __forceinline__ int operand_row(const int* rowmap, int base, int n) {
  return rowmap ? rowmap[base + n] : base + n;
}

// Operand rows of one item (x, or h as hi + lo) and their per-64-group sums by
// 16-byte cp.async (all threads).  The sums go through L2 only: they may have
// been written by another CTA of the same kernel, next to sums this SM already
// read, so an L1-allocating copy could return a stale line.
__device__ __forceinline__ void stage_operand_async(const TileGeo& t, int c, const int* rowmap,
                                                    int base, int ntok, const uint16_t* B,
                                                    const uint16_t* Blo, const float* Bsum,
                                                    uint8_t* st, const StageLayout& L) {
  const int tid = threadIdx.x;
  const int cpt = (t.CK * 2) >> 4;
  const int nparts = Blo ? 2 : 1;
  for (int i = tid; i < nparts * ntok * cpt; i += kUnitThreads) {
    const int part = i / (ntok * cpt);
    const int ii = i - part * ntok * cpt;
    const int n = ii / cpt, q = ii - n * cpt;
    const uint16_t* src =
        (part ? Blo : B) + (size_t)operand_row(rowmap, base, n) * t.K + (size_t)c * t.CK;
    cp_async16(st + (part ? L.xlo : L.x) + n * L.bpitch + q * 16,
               reinterpret_cast<const uint8_t*>(src) + q * 16);
  }
  const int ng = t.ng;
  const int ksw = t.K / 64;
  if ((ng & 3) == 0) {
    const int spt = ng >> 2;
    for (int i = tid; i < ntok * spt; i += kUnitThreads) {
      const int n = i / spt, q = i - n * spt;
      cp_async16(st + L.xsum + (n * ng + 4 * q) * 4,
                 Bsum + (size_t)operand_row(rowmap, base, n) * ksw + (size_t)c * ng + 4 * q);
    }
  } else {
    for (int i = tid; i < ntok * ng; i += kUnitThreads) {
      const int n = i / ng, q = i - n * ng;
      reinterpret_cast<float*>(st + L.xsum)[n * ng + q] =
          __ldcg(Bsum + (size_t)operand_row(rowmap, base, n) * ksw + (size_t)c * ng + q);
    }
  }
}

// Same staging with plain L2 loads (operands produced inside the same kernel,
// copied after their ready counter was observed).
__device__ __forceinline__ void stage_operand_sync(const TileGeo& t, int c, const int* rowmap,
                                                   int base, int ntok, const uint16_t* B,
                                                   const uint16_t* Blo, const float* Bsum,
                                                   uint8_t* st, const StageLayout& L) {
  const int tid = threadIdx.x;
  const int cpt = (t.CK * 2) >> 4;
  const int nparts = Blo ? 2 : 1;
  for (int i = tid; i < nparts * ntok * cpt; i += kUnitThreads) {
    const int part = i / (ntok * cpt);
    const int ii = i - part * ntok * cpt;
    const int n = ii / cpt, q = ii - n * cpt;
    const uint16_t* src =
        (part ? Blo : B) + (size_t)operand_row(rowmap, base, n) * t.K + (size_t)c * t.CK;
    const uint4 v = __ldcg(reinterpret_cast<const uint4*>(src) + q);
    *reinterpret_cast<uint4*>(st + (part ? L.xlo : L.x) + n * L.bpitch + q * 16) = v;
  }
  const int ng = t.ng;
  const int ksw = t.K / 64;
  for (int i = tid; i < ntok * ng; i += kUnitThreads) {
    const int n = i / ng, q = i - n * ng;
    reinterpret_cast<float*>(st + L.xsum)[n * ng + q] =
        __ldcg(Bsum + (size_t)operand_row(rowmap, base, n) * ksw + (size_t)c * ng + q);
  }
}

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

// One k-chunk of one warp over its 16-row tile and the staged operand tokens
// (n < ntok), added into acc.  acc[0]: (row g, token 2t), acc[1]: (g, 2t+1),
// acc[2]: (g+8, 2t), acc[3]: (g+8, 2t+1).
template <int FMT, bool F16A, bool SPLIT>
__device__ __forceinline__ void compute_pass(const TileGeo& tg, const uint8_t* st,
                                             const StageLayout& L, int ntok, float (&acc)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, t = lane & 3;
  const int ng = tg.ng;
  const uint8_t* codes = st + L.a + warp * ng * (FMT == MOE_FMT_AFFINE3_G64 ? 384 : 512);
  const uint8_t* scales = st + L.a + tg.code_bytes;
  const float* xs = reinterpret_cast<const float*>(st + L.xsum);
  const bool bv = gq < ntok;
  const bool c0 = 2 * t < ntok, c1 = 2 * t + 1 < ntok;
  const uint8_t* xrow = st + L.x + gq * L.bpitch + 32 * t;
  const uint8_t* xlrow = st + L.xlo + gq * L.bpitch + 32 * t;
#pragma unroll 2
  for (int G = 0; G < ng; ++G) {
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
    uint32_t bf[8];
    if (bv) {
      const uint4 x0 = *reinterpret_cast<const uint4*>(xrow + G * 128);
      const uint4 x1 = *reinterpret_cast<const uint4*>(xrow + G * 128 + 16);
      bf[0] = x0.x; bf[1] = x0.y; bf[2] = x0.z; bf[3] = x0.w;
      bf[4] = x1.x; bf[5] = x1.y; bf[6] = x1.z; bf[7] = x1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) bf[i] = 0u;
    }
    // k-step m uses word (m < 2 ? w0/w2 : w1/w3) nibble pairs (2(m&1), +4)
    // and (2(m&1)+1, +5) of rows g and g+8
    const uint32_t A00 = code_pair<F16A>(w0), A01 = code_pair<F16A>(w2);
    const uint32_t A02 = code_pair<F16A>(w0 >> 4), A03 = code_pair<F16A>(w2 >> 4);
    const uint32_t A10 = code_pair<F16A>(w0 >> 8), A11 = code_pair<F16A>(w2 >> 8);
    const uint32_t A12 = code_pair<F16A>(w0 >> 12), A13 = code_pair<F16A>(w2 >> 12);
    const uint32_t A20 = code_pair<F16A>(w1), A21 = code_pair<F16A>(w3);
    const uint32_t A22 = code_pair<F16A>(w1 >> 4), A23 = code_pair<F16A>(w3 >> 4);
    const uint32_t A30 = code_pair<F16A>(w1 >> 8), A31 = code_pair<F16A>(w3 >> 8);
    const uint32_t A32 = code_pair<F16A>(w1 >> 12), A33 = code_pair<F16A>(w3 >> 12);
    // two MMA chains (k-steps 0,2 and 1,3), summed once
    float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
    mma16816<F16A>(e0, A00, A01, A02, A03, bf[0], bf[1]);
    mma16816<F16A>(e1, A10, A11, A12, A13, bf[2], bf[3]);
    mma16816<F16A>(e0, A20, A21, A22, A23, bf[4], bf[5]);
    mma16816<F16A>(e1, A30, A31, A32, A33, bf[6], bf[7]);
    if constexpr (SPLIT) {
      if (bv) {
        const uint4 x0 = *reinterpret_cast<const uint4*>(xlrow + G * 128);
        const uint4 x1 = *reinterpret_cast<const uint4*>(xlrow + G * 128 + 16);
        bf[0] = x0.x; bf[1] = x0.y; bf[2] = x0.z; bf[3] = x0.w;
        bf[4] = x1.x; bf[5] = x1.y; bf[6] = x1.z; bf[7] = x1.w;
      }
      mma16816<F16A>(e0, A00, A01, A02, A03, bf[0], bf[1]);
      mma16816<F16A>(e1, A10, A11, A12, A13, bf[2], bf[3]);
      mma16816<F16A>(e0, A20, A21, A22, A23, bf[4], bf[5]);
      mma16816<F16A>(e1, A30, A31, A32, A33, bf[6], bf[7]);
    }
    float s0, s1, b0, b1;
    if constexpr (FMT == MOE_FMT_W4A16_SYM_G128) {
      const uint32_t sv =
          *reinterpret_cast<const uint32_t*>(scales + (((warp * (ng >> 1)) + (G >> 1)) * 8 + gq) * 4);
      s0 = half_bits_to_float(uint16_t(sv & 0xFFFFu));
      s1 = half_bits_to_float(uint16_t(sv >> 16));
      b0 = -8.f * s0;
      b1 = -8.f * s1;
    } else {
      const uint2 sv = *reinterpret_cast<const uint2*>(scales + ((warp * ng + G) * 8 + gq) * 8);
      s0 = half_bits_to_float(uint16_t(sv.x & 0xFFFFu));
      b0 = half_bits_to_float(uint16_t(sv.x >> 16));
      s1 = half_bits_to_float(uint16_t(sv.y & 0xFFFFu));
      b1 = half_bits_to_float(uint16_t(sv.y >> 16));
    }
    if constexpr (!F16A) {  // operand codes carry +128
      b0 = fmaf(-128.f, s0, b0);
      b1 = fmaf(-128.f, s1, b1);
    }
    const float X0 = c0 ? xs[(2 * t) * ng + G] : 0.f;
    const float X1 = c1 ? xs[(2 * t + 1) * ng + G] : 0.f;
    const float d0 = e0[0] + e1[0], d1 = e0[1] + e1[1];
    const float d2 = e0[2] + e1[2], d3 = e0[3] + e1[3];
    acc[0] = fmaf(s0, d0, acc[0]);
    acc[0] = fmaf(b0, X0, acc[0]);
    acc[1] = fmaf(s0, d1, acc[1]);
    acc[1] = fmaf(b0, X1, acc[1]);
    acc[2] = fmaf(s1, d2, acc[2]);
    acc[2] = fmaf(b1, X0, acc[2]);
    acc[3] = fmaf(s1, d3, acc[3]);
    acc[3] = fmaf(b1, X1, acc[3]);
  }
}

// Where a down unit's results go: y[o * H + row] with o = out_idx[p] for
// bucket position p (the assignment id), or o = p (shared expert: the token).
struct Sink {
  float* out;
  const int* out_idx;  // nullptr: identity
  int rows;            // H
};

__device__ __forceinline__ void write_down(const Sink& sk, const Unit& u, const float (&acc)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, t = lane & 3;
  const int row = u.blk * kUnitRows + 16 * warp + gq;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int n = 2 * t + h;
    if (n < u.cnt) {
      const int p = u.off + n;
      const int o = sk.out_idx ? __ldcg(sk.out_idx + p) : p;
      float* dst = sk.out + (size_t)o * sk.rows + row;
      dst[0] = acc[h];
      dst[8] = acc[2 + h];
    }
  }
}

// SwiGLU epilogue of a gate/up unit (all threads): warps 0..3 hold the gate
// sums of rows 64j + 16w + {g, g+8}, warps 4..7 the matching up sums.
//   h = a / (1 + exp(-a)) * u,  hi = bf16(h), lo = bf16(h - hi)
// stored k-permuted at bucket position off + n, and hsum[off + n][j] =
// sum over the 64 rows of (hi + lo) in a fixed tree (8 rows by shuffles,
// then the 4 warps in order).
struct EpiSmem {
  float up[4][32][4];
  float red[4][8];
};

__device__ __forceinline__ void swiglu_epilogue(const float (&acc)[4], EpiSmem& E, const Unit& u,
                                                int inter, uint16_t* hh, uint16_t* hl,
                                                float* hsum, float* hout) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, t = lane & 3;
  if (warp >= 4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) E.up[warp - 4][lane][i] = acc[i];
  }
  __syncthreads();
  if (warp < 4) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (i < 2 ? gq : gq + 8);
      const int n = 2 * t + (i & 1);
      const float a = acc[i];
      const float h = a / (1.f + expf(-a)) * E.up[warp][lane][i];
      const __nv_bfloat16 hi = __float2bfloat16_rn(h);
      const __nv_bfloat16 lo = __float2bfloat16_rn(h - __bfloat162float(hi));
      const float c = __bfloat162float(hi) + __bfloat162float(lo);
      if (n < u.cnt) {
        const size_t p = (size_t)(u.off + n);
        const int j = u.blk * 64 + 16 * warp + r;
        hh[p * inter + kperm_pos(j)] = __bfloat16_as_ushort(hi);
        hl[p * inter + kperm_pos(j)] = __bfloat16_as_ushort(lo);
        if (hout) hout[p * inter + j] = h;
      }
      if (i & 1)
        s1 += c;
      else
        s0 += c;
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, o);
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    }
    if (gq == 0) {
      E.red[warp][2 * t] = s0;
      E.red[warp][2 * t + 1] = s1;
    }
  }
  __syncthreads();
  if (tid < u.cnt)
    hsum[(size_t)(u.off + tid) * (inter / 64) + u.blk] =
        ((E.red[0][tid] + E.red[1][tid]) + E.red[2][tid]) + E.red[3][tid];
}

// Sub-slot table: sub-slot ss holds tokens [off, off + cnt) of expert e, in
// bucket positions (routed) -- or, for a fixed expert over T tokens (shared
// expert, single-expert MLP), sub-slot ss is tokens [8 ss, min(T, 8 ss + 8)).
struct SubSlots {
  const int* n;      // device count (nullptr: fixed expert)
  const int* e;
  const int* off;
  const int* cnt;
  int fixed_e;
  int fixed_T;
};

__device__ __forceinline__ int subslot_count(const SubSlots& S) {
  return S.n ? __ldcg(S.n) : (S.fixed_T + kMaxTok - 1) / kMaxTok;
}

__device__ __forceinline__ void subslot_get(const SubSlots& S, int ss, int& e, int& off,
                                            int& cnt) {
  if (S.n) {
    e = __ldcg(S.e + ss);
    off = __ldcg(S.off + ss);
    cnt = __ldcg(S.cnt + ss);
  } else {
    e = S.fixed_e;
    off = kMaxTok * ss;
    cnt = min(kMaxTok, S.fixed_T - kMaxTok * ss);
  }
}

// Operand rows of a unit kind: row of token slot n of a pass starting at
// bucket position `base` is rowmap[base + n] (or base + n without a map).
struct OperandSrc {
  const uint16_t* B;
  const uint16_t* Blo;
  const float* Bsum;
  const int* rowmap;
};

// Weighted combine of one 128-row block of the output for all T tokens:
//   out[t, h] = round( sum_j w[t, j] * y[t*k + j, h]  +  s_t * ysh[t, h] )
// an fp32 fma chain in slot order with the shared slot last; y and ysh are
// summed over their k-chunk planes first (in chunk order).
struct CombineArgs {
  const float* y;      // [nchd][T*k][H]
  const float* w;      // [T][k]
  const float* ysh;    // [nchd][T][H] or nullptr
  const float* sg;     // [T] or nullptr (weight 1)
  uint16_t* out;       // [T][H]
  int nchd, T, k, H, f16;
};

__device__ __forceinline__ void combine_block(const CombineArgs& A, int rb, int t0, int t1) {
  const int P = A.T * A.k;
  for (int i = threadIdx.x; i < (t1 - t0) * kUnitRows; i += blockDim.x) {
    const int t = t0 + i / kUnitRows;
    const int h = rb * kUnitRows + (i % kUnitRows);
    float acc = 0.f;
    for (int j = 0; j < A.k; ++j) {
      const int a = t * A.k + j;
      float v = 0.f;
      for (int c = 0; c < A.nchd; ++c) v += __ldcg(A.y + ((size_t)c * P + a) * A.H + h);
      acc = fmaf(__ldcg(A.w + a), v, acc);
    }
    if (A.ysh) {
      float v = 0.f;
      for (int c = 0; c < A.nchd; ++c) v += __ldcg(A.ysh + ((size_t)c * A.T + t) * A.H + h);
      acc = fmaf(A.sg ? __ldcg(A.sg + t) : 1.f, v, acc);
    }
    A.out[(size_t)t * A.H + h] = float_to_act_bits(acc, A.f16 != 0);
  }
}

// Copy-free x preparation: row t of x -> k-permuted copy and per-64-group
// sums.  One warp per (t, group); `task` enumerates them.
__device__ __forceinline__ void xprep_task(const uint16_t* x, int H, int f16, uint16_t* xperm,
                                           float* xsum, int task) {
  const int lane = threadIdx.x & 31;
  const int ng = H >> 6;
  const int t = task / ng, G = task - t * ng;
  const int j0 = G * 64 + 2 * lane;
  const size_t rb = (size_t)t * H;
  const uint32_t v = *reinterpret_cast<const uint32_t*>(x + rb + j0);
  const uint16_t v0 = uint16_t(v & 0xFFFFu), v1 = uint16_t(v >> 16);
  xperm[rb + kperm_pos(j0)] = v0;
  xperm[rb + kperm_pos(j0 + 1)] = v1;
  float s = act_to_float(v0, f16 != 0) + act_to_float(v1, f16 != 0);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) xsum[(size_t)t * ng + G] = s;
}

}  // namespace moe
