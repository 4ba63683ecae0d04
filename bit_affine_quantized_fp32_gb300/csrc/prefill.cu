// prefill.cu -- the expert GEMMs of a prefill window on tcgen05.
//
// For T > 32 tokens an expert sees up to hundreds of rows, so its weights are
// dequantised once per tile of kPfTile rows and fed to the tensor cores:
// D[128 weight rows x N tokens] += A[128 x 128] * B[N x 128]^T per stage of
// 128 columns (two 64-column code groups, eight K16 MMAs behind one
// hand-off), fp16 operands, fp32 accumulators in tensor memory.  A (the
// dequantised weights) is written straight into tensor memory; B (the
// activation rows) is staged in shared memory.
// One persistent CTA per SM, 18 warps:
//   warps 0-3   epilogue: tensor memory -> registers, 32 columns a load
//               (thread = accumulator lane = weight row), SwiGLU -> fp16 h
//               (mode 0; the fast exponential and division, a few ulp of
//               fp32, far below the fp16 rounding of h) or fp32 y rows
//               (mode 1);
//   warps 4-11  dequantisation: one weight item (128 rows x CK columns, the
//               kernel-tiled layout) per raw stage, two 64-column groups at
//               a time into a tensor-memory A stage: w = fp16(s * q + b), one
//               fused multiply-add of the fp16 scale, the exact code and the
//               fp16 bias (W4A16: s * u - 8 s), rounded once;
//   warp 12     TMA bulk copies of the raw weight items (2 stages);
//   warp 13     allocates tensor memory and issues the MMAs (one thread);
//               tcgen05.commit frees A/B stages and hands accumulators over;
//   warps 14-17 the operand rows of each stage into a B stage, 32 rows a
//               warp (cp.async of 16-byte pieces; one instruction copies 4
//               whole 128-byte rows of a 64-column half): fp16 x rows
//               (mode 0) or fp16 h rows (mode 1).
// A stage is complete when the eight dequantisation warps and the 128 copy
// threads have arrived on its barrier (one wait for the MMA thread).
// Dequantisation warp w takes M-tile w of the block and places it at
// tensor-memory lanes 32 (w % 4) + 16 (w / 4) .. + 15, inside its own lane
// quarter: in mode 0 (gate tiles 0-3, the matching up tiles 4-7) each
// epilogue warp then holds 16 gate rows and their 16 up rows and pairs them
// with one shuffle.  A lane's four code words (rows g, g + 8; 16 columns
// each) are transposed within its quad so that the 16x256b tensor-memory
// stores put every element at its own column (the packed layout keeps 16
// consecutive columns per lane; the store shape wants 4 runs of 4).
// B stages hold two 64-column halves in the K-major 128-byte-swizzled layout
// (umma.cuh): the row copies write one shared-memory wavefront per quarter
// warp.
// One MMA per 16 columns.  The activations enter as fp16: bf16 x is converted
// once per call (exact in fp16's normal range; a value beyond it sets
// MOE_ERR_RANGE), and h is stored as fp16 (likewise checked).  Two
// accumulators of kPfTile columns let the epilogue of one unit overlap the
// MMAs of the next.  Every wait is bounded (the workspace's limit, then the
// status word gets MOE_ERR_TIMEOUT and the remaining waits return at once);
// the dequantisation and MMA roles poll, the long waits of the copy and
// epilogue roles let the hardware suspend the warp.
//
// Sources: "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803"
// (prefill windows through grouped expert GEMMs, SwiGLU epilogue).

#include "prefill.h"
#include "host.h"
#include "engine.cuh"
#include "umma.cuh"

namespace moe {

namespace {

constexpr int kPfRaw = 2;                    // raw weight-item stages
constexpr int kPfGrp = 64;                   // columns per code group / swizzle half
constexpr int kPfKBlk = 2 * kPfGrp;          // columns per stage (8 x K16)
constexpr int kPfHalf = kPfTile * kPfGrp * 2;  // one 64-column half of a B stage
constexpr int kPfB = 2 * kPfHalf;            // B stage: kPfTile rows x 128 fp16
constexpr int kPfStages = 4;                 // A/B stages
constexpr int kPfRawWarp = 12, kPfMmaWarp = 13, kPfBWarp0 = 14, kPfBWarps = 4;
static_assert((kPfBWarp0 + kPfBWarps) * 32 == kPfThreads, "warp roles cover the block");
static_assert(kPfBWarps * 32 == kPfTile, "one B warp per 32 tile rows");
// tensor memory: two accumulators of kPfTile fp32 columns, then the A stages
// (128 fp16 columns = 64 columns each)
constexpr int kPfACol0 = 2 * kPfTile;
constexpr int kPfACols = kPfKBlk / 2;
constexpr int kPfTmemCols = 512;
static_assert(kPfACol0 + kPfStages * kPfACols <= kPfTmemCols, "tensor memory budget");
__host__ __device__ constexpr int pf_stages(int mode) { return (void)mode, kPfStages; }
__host__ __device__ constexpr int pf_stage_bytes(int mode) { return (void)mode, kPfB; }

__host__ __device__ inline int raw_stage_bytes(const TileGeo& g) {
  return (g.item_bytes + 1023) & ~1023;
}

struct PfSmem {
  uint64_t raw_full[kPfRaw], raw_empty[kPfRaw];
  uint64_t full[kPfStages], ab_empty[kPfStages];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem;
  WaitCtl wc;
};

struct PfUnit {
  int e, off, cnt, m;
  bool sh;  // a unit of the second (shared-expert) bank
};

__device__ __forceinline__ int pf_tiles(const PrefillJob& J) {
  return J.n_tiles ? __ldcg(J.n_tiles) : (J.fixed_T + kPfTile - 1) / kPfTile;
}

// units of the second bank (they come first)
__device__ __forceinline__ int pf_sh_units(const PrefillJob& J) {
  return J.sh_base ? (J.sh_T + kPfTile - 1) / kPfTile * J.g.nblk : 0;
}

__device__ __forceinline__ PfUnit pf_unit(const PrefillJob& J, int u) {
  const int nblk = J.g.nblk;
  const int nsh = pf_sh_units(J);
  PfUnit r;
  r.sh = u < nsh;
  if (r.sh) {
    const int t = u / nblk;
    r.m = u - t * nblk;
    r.e = 0;
    r.off = kPfTile * t;
    r.cnt = min(kPfTile, J.sh_T - kPfTile * t);
    return r;
  }
  u -= nsh;
  const int t = u / nblk;
  r.m = u - t * nblk;
  if (J.n_tiles) {
    r.e = __ldcg(J.te + t);
    r.off = __ldcg(J.toff + t);
    r.cnt = __ldcg(J.tcnt + t);
  } else {
    r.e = J.fixed_e;
    r.off = kPfTile * t;
    r.cnt = min(kPfTile, J.fixed_T - kPfTile * t);
  }
  return r;
}

// One 8-code word (codes in nibble order [0 2 4 6 1 3 5 7]) -> 8 fp16 weights
// in column order: w = fma(s, q, b) in fp16 (the exact value rounded once;
// q is exact as 1024 + q - 1024).
__device__ __forceinline__ uint4 dequant_word16(uint32_t w, __half2 s2, __half2 b2) {
  const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  uint32_t h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t p;
    asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;\n" : "=r"(p) : "r"(w >> (4 * j)));
    const __half2 q = __hsub2(*reinterpret_cast<__half2*>(&p), k1024);
    const __half2 v = __hfma2(s2, q, b2);
    h[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}

// Accumulator lane (A row) of row i of M-tile w: lanes 32 (w % 4) + 16 (w / 4)
// + i, in the lane quarter of dequantisation warp 4 + w.  In mode 0 the gate
// tile w (w < 4) and its up tile w + 4 share quarter w.
__device__ __forceinline__ int pf_arow(int w, int i) { return 32 * (w & 3) + 16 * (w >> 2) + i; }

// Quad transpose of one row's codes.  Lane t of a quad holds the row's
// 4-code blocks 4t .. 4t + 3 (of the 16 in a 64-column group): Wa blocks 4t,
// 4t + 1 and Wb blocks 4t + 2, 4t + 3, block 2i + p of a word in its bytes p
// and p + 2 (the nibble order of the packed words).  Afterwards Na holds
// blocks t, 4 + t and Nb blocks 8 + t, 12 + t in the same word format.
// Round r brings lane t the word of lane t ^ r that holds block 4 (t ^ r) + t.
__device__ __forceinline__ void quad_transpose(uint32_t Wa, uint32_t Wb, int t, uint32_t& Na,
                                               uint32_t& Nb) {
  const bool hi = t >= 2;
  uint32_t v[4];
  v[0] = hi ? Wb : Wa;
#pragma unroll
  for (int r = 1; r < 4; ++r) v[r] = __shfl_xor_sync(0xffffffffu, ((t ^ r) >= 2) ? Wb : Wa, r);
  // v[r] holds block 4 (t ^ r) + t in bytes p, p + 2 (p = t & 1); it goes to
  // word (t ^ r) / 2 at position (t ^ r) & 1
  const uint32_t sel = (t & 1) ? 0x3715u : 0x6240u;
  uint32_t X, Y;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(X) : "r"(v[0]), "r"(v[1]), "r"(sel));
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(Y) : "r"(v[2]), "r"(v[3]), "r"(sel));
  Na = hi ? Y : X;
  Nb = hi ? X : Y;
}

// Group G of the raw item into the 32 tensor-memory columns at ta (lane
// field: the tile's first lane): thread (tile w, lane l = 4 g + t) converts
// the codes of tile rows g and g + 8 -- after the quad transpose, columns
// 16 j + 4 t .. + 3 (j = 0..3) -- and stores them with four 16x256b stores
// (store j: columns 8 j .. 8 j + 7, two fp16 a column).
template <int FMT>
__device__ __forceinline__ void dequant_group(const TileGeo& g, const uint8_t* raw, int G,
                                              uint32_t ta, int w, int l) {
  const int NG = g.ng;
  const int gq = l >> 2, t = l & 3;
  uint32_t W0, W1, W2, W3;
  if constexpr (FMT == MOE_FMT_AFFINE3_G64) {
    const uint32_t* pl = reinterpret_cast<const uint32_t*>(raw + (w * NG + G) * 384) + l;
    planes_to_words(pl[0], pl[32], pl[64], W0, W1, W2, W3);
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(raw + (w * NG + G) * 512 + l * 16);
    W0 = v.x;
    W1 = v.y;
    W2 = v.z;
    W3 = v.w;
  }
  const uint8_t* sc = raw + g.code_bytes;
  __half s0, s1, b0, b1;
  if constexpr (FMT == MOE_FMT_W4A16_SYM_G128) {
    const uint32_t sv =
        *reinterpret_cast<const uint32_t*>(sc + ((w * 8 + gq) * (NG / 2) + (G >> 1)) * 4);
    s0 = __ushort_as_half(uint16_t(sv & 0xFFFF));
    s1 = __ushort_as_half(uint16_t(sv >> 16));
    // w = s (u - 8) for the stored nibble u: fma(s, u, -8 s), -8 s exact
    b0 = __hmul(s0, __ushort_as_half(0xC800));
    b1 = __hmul(s1, __ushort_as_half(0xC800));
  } else {
    const uint2 sv = *reinterpret_cast<const uint2*>(sc + ((w * 8 + gq) * NG + G) * 8);
    s0 = __ushort_as_half(uint16_t(sv.x & 0xFFFF));
    b0 = __ushort_as_half(uint16_t(sv.x >> 16));
    s1 = __ushort_as_half(uint16_t(sv.y & 0xFFFF));
    b1 = __ushort_as_half(uint16_t(sv.y >> 16));
  }
  const __half2 s02 = __halves2half2(s0, s0), s12 = __halves2half2(s1, s1);
  const __half2 b02 = __halves2half2(b0, b0), b12 = __halves2half2(b1, b1);
  uint32_t N0, N1, N2, N3;
  quad_transpose(W0, W1, t, N0, N1);  // row g
  quad_transpose(W2, W3, t, N2, N3);  // row g + 8
  const uint4 q0 = dequant_word16(N0, s02, b02), q1 = dequant_word16(N1, s02, b02);
  const uint4 q2 = dequant_word16(N2, s12, b12), q3 = dequant_word16(N3, s12, b12);
  tmem_st_16x256b(ta + 0, q0.x, q0.y, q2.x, q2.y);
  tmem_st_16x256b(ta + 8, q0.z, q0.w, q2.z, q2.w);
  tmem_st_16x256b(ta + 16, q1.x, q1.y, q3.x, q3.y);
  tmem_st_16x256b(ta + 24, q1.z, q1.w, q3.z, q3.w);
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}

template <int FMT, int MODE>
__global__ void __launch_bounds__(kPfThreads, 1) k_prefill(const __grid_constant__ PrefillJob J) {
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  __shared__ PfSmem S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const TileGeo& g = J.g;
  constexpr int NS = pf_stages(MODE), SB = pf_stage_bytes(MODE);
  const int RB = raw_stage_bytes(g);
  // the swizzled stages need 1024-byte alignment (the launch adds the slack)
  uint8_t* smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
  uint8_t* raw = smem;
  uint8_t* stages = smem + kPfRaw * RB;  // B stage s at s * kPfB; RB a multiple of 1024
  if (tid == 0) {
    for (int i = 0; i < kPfRaw; ++i) {
      mbar_init(&S.raw_full[i], 1);
      mbar_init(&S.raw_empty[i], 8);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&S.full[i], 8 + 32 * kPfBWarps);  // dequantisation warps + copy threads
      mbar_init(&S.ab_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.acc_full[i], 1);
      mbar_init(&S.acc_empty[i], 4);
    }
    wait_ctl_init(S.wc, J.status);
  }
  if (warp == kPfMmaWarp) tmem_alloc(&S.tmem, kPfTmemCols);
  fence_proxy_async();
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tbase = S.tmem;
  const int nunits = pf_sh_units(J) + pf_tiles(J) * g.nblk;
  const int G = gridDim.x;
  const int NG = g.ng, nch = g.nch, nks = nch * NG / 2;  // stages per unit
  int* status = J.status;

  if (warp == kPfRawWarp) {
    // ---- raw weight items
    int ri = 0;
    for (int u = blockIdx.x; u < nunits; u += G) {
      const PfUnit U = pf_unit(J, u);
      for (int c = 0; c < nch; ++c, ++ri) {
        const int rs = ri % kPfRaw;
        if (lane == 0) {
          if (ri >= kPfRaw) {
            mbar_wait_bounded(&S.raw_empty[rs], ((ri / kPfRaw) - 1) & 1, &S.wc, status, true);
            // the stage's previous copy has landed (immediate unless a timeout
            // let the consumers skip their wait): one copy per barrier phase
            mbar_drain(&S.raw_full[rs], ((ri / kPfRaw) - 1) & 1);
          }
          mbar_expect_tx(&S.raw_full[rs], unsigned(g.item_bytes));
          bulk_g2s(raw + rs * RB,
                   (U.sh ? J.sh_base : J.base) + (size_t)U.e * g.expert_bytes +
                       (size_t)(U.m * nch + c) * g.item_bytes,
                   unsigned(g.item_bytes), &S.raw_full[rs]);
        }
        __syncwarp();
      }
    }
    // the last copies have landed before the CTA may exit, also after a timeout
    if (lane == 0)
      for (int i = max(0, ri - kPfRaw); i < ri; ++i)
        mbar_drain(&S.raw_full[i % kPfRaw], (i / kPfRaw) & 1);
  } else if (warp >= kPfBWarp0) {
    // ---- operand rows, one 64-column group per stage.  B warp b owns tile
    // rows 32 b .. 32 b + 31; instruction i copies rows 32 b + 4 i .. + 3,
    // lane l piece l % 8 of row 32 b + 4 i + l / 8; the row addresses are
    // resolved once per unit.
    const int bw = warp - kPfBWarp0;
    const int pc = lane & 7;
    int ks = 0;
    for (int u = blockIdx.x; u < nunits; u += G) {
      const PfUnit U = pf_unit(J, u);
      const uint16_t* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int n = 32 * bw + 4 * i + (lane >> 3);
        const int row =
            n < U.cnt ? ((MODE == 0 && J.gather && !U.sh) ? __ldg(J.perm + U.off + n) / J.k
                                                          : U.off + n)
                      : 0;
        src[i] = (U.sh ? J.sh_B : J.B) + (size_t)row * J.ldB + 8 * pc;
      }
      for (int q = 0; q < nks; ++q, ++ks) {
        const int s = ks % NS;
        if (ks >= NS)
          mbar_wait_bounded(&S.ab_empty[s], ((ks / NS) - 1) & 1, &S.wc, status, true);
        const int k0 = q * kPfKBlk;
        uint8_t* B = stages + s * SB;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int n = 32 * bw + 4 * i + (lane >> 3);
            if (n < U.cnt)
              cp_async16(B + h * kPfHalf + umma_off_sw128(n, 8 * pc), src[i] + k0 + kPfGrp * h);
          }
        cp_async_arrive_noinc(&S.full[s]);
      }
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");
  } else if (warp == kPfMmaWarp) {
    // ---- MMA issue (one thread)
    if (lane == 0) {
      int ks = 0, ui = 0;
      for (int u = blockIdx.x; u < nunits; u += G, ++ui) {
        const PfUnit U = pf_unit(J, u);
        const int a = ui & 1;
        if (ui >= 2) mbar_wait_bounded(&S.acc_empty[a], ((ui >> 1) - 1) & 1, &S.wc, status);
        tmem_fence_after();
        const int N = max(16, (U.cnt + 15) & ~15);
        const uint32_t idesc = umma_idesc_f16(128, N);
        const uint32_t d = tbase + uint32_t(a * kPfTile);
        for (int q = 0; q < nks; ++q, ++ks) {
          const int s = ks % NS;
          mbar_wait_bounded(&S.full[s], (ks / NS) & 1, &S.wc, status);
          fence_proxy_async();  // the cp.async rows of B
          tmem_fence_after();   // the tensor-memory stores of A
          const uint32_t ta = tbase + uint32_t(kPfACol0 + s * kPfACols);
          const uint32_t ba = smem_u32(stages + s * SB);
#pragma unroll
          for (int kk = 0; kk < kPfKBlk / 16; ++kk)
            umma_f16_tmem_a(d, ta + 8 * kk,
                            umma_desc_sw128(ba + (kk >> 2) * kPfHalf + 32 * (kk & 3)), idesc,
                            q > 0 || kk > 0);
          umma_commit(&S.ab_empty[s]);
        }
        umma_commit(&S.acc_full[a]);
      }
      // every MMA has completed before tensor memory is released, also after
      // a timeout: the last commit arrives once all earlier MMAs are done
      if (ui > 0) mbar_drain(&S.acc_full[(ui - 1) & 1], ((ui - 1) >> 1) & 1);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- dequantisation: warp 4 + w takes M-tile w
    const int w = warp - 4;
    const uint32_t tw = tbase + (uint32_t(pf_arow(w, 0)) << 16);
    int ri = 0, ks = 0;
    for (int u = blockIdx.x; u < nunits; u += G) {
      const PfUnit U = pf_unit(J, u);
      (void)U;
      for (int c = 0; c < nch; ++c, ++ri) {
        const int rs = ri % kPfRaw;
        mbar_wait_bounded(&S.raw_full[rs], (ri / kPfRaw) & 1, &S.wc, status);
        for (int Gi = 0; Gi < NG; Gi += 2, ++ks) {
          const int s = ks % NS;
          if (ks >= NS) mbar_wait_bounded(&S.ab_empty[s], ((ks / NS) - 1) & 1, &S.wc, status);
          const uint32_t ta = tw + uint32_t(kPfACol0 + s * kPfACols);
          dequant_group<FMT>(g, raw + rs * RB, Gi, ta, w, lane);
          dequant_group<FMT>(g, raw + rs * RB, Gi + 1, ta + kPfGrp / 2, w, lane);
          tmem_wait_st();
          tmem_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.full[s]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.raw_empty[rs]);
      }
    }
  } else {
    // ---- epilogue: thread (warp q, lane l) = accumulator lane 32 q + l
    int ui = 0;
    for (int u = blockIdx.x; u < nunits; u += G, ++ui) {
      const PfUnit U = pf_unit(J, u);
      const int a = ui & 1;
      mbar_wait_bounded(&S.acc_full[a], (ui >> 1) & 1, &S.wc, status, true);
      tmem_fence_after();
      const uint32_t tl = tbase + (uint32_t(32 * warp) << 16) + uint32_t(a * kPfTile);
      for (int c0 = 0; c0 < U.cnt; c0 += 32) {
        if (MODE == 0) {
          // lanes 0-15: gate rows 64 m + 16 q + l, lanes 16-31 the matching
          // up rows; lane l < 16 finishes tokens c0 .. c0 + 15 of its
          // column, lane l + 16 tokens c0 + 16 .. c0 + 31
          float v[32];
          tmem_ld32(tl + uint32_t(c0), v);
          const bool hi = lane >= 16;
          const size_t col = 64 * size_t(U.m) + 16 * warp + (lane & 15);
          uint16_t* hout = U.sh ? J.sh_h : J.h;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const float recv = __shfl_xor_sync(0xffffffffu, hi ? v[jj] : v[16 + jj], 16);
            const float ga = hi ? recv : v[jj];
            const float up = hi ? v[16 + jj] : recv;
            const int n = c0 + jj + (hi ? 16 : 0);
            if (n < U.cnt) {
              const float hv = __fdividef(ga, 1.f + __expf(-ga)) * up;
              hout[(size_t)(U.off + n) * J.ldh + col] = __half_as_ushort(__float2half_rn(hv));
              if (!(fabsf(hv) <= 65504.f)) atomicExch(status, int(MOE_ERR_RANGE));
            }
          }
        } else {
          // output rows of tokens c0 .. c0 + 31, one per lane, then two
          // 64-byte row pieces a token
          const int nl = c0 + lane;
          const int orow =
              nl < U.cnt ? ((J.scatter && !U.sh) ? __ldg(J.perm + U.off + nl) : U.off + nl) : 0;
          float v[32];
          tmem_ld32(tl + uint32_t(c0), v);
          // lane 32 q + l holds row l % 16 of M-tile q + 4 (l / 16)
          const size_t col = 128 * size_t(U.m) + 16 * (warp + 4 * (lane >> 4)) + (lane & 15);
          float* yout = U.sh ? J.sh_y : J.y;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int row = __shfl_sync(0xffffffffu, orow, j);
            if (c0 + j < U.cnt) yout[(size_t)row * J.ldy + col] = v[j];
          }
        }
      }
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acc_empty[a]);
    }
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  if (warp == kPfMmaWarp) tmem_dealloc(tbase, kPfTmemCols);
}

template <int FMT, int MODE>
cudaError_t launch_t(const PrefillJob& J, int sms, cudaStream_t st) {
  const int smem = prefill_smem(J.g, MODE);
  if (smem <= 0) return cudaErrorInvalidValue;
  const cudaError_t e = ensure_dynamic_smem((const void*)k_prefill<FMT, MODE>, smem);
  if (e != cudaSuccess) return e;
  k_prefill<FMT, MODE><<<sms, kPfThreads, smem, st>>>(J);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_fmt(const PrefillJob& J, int mode, int sms, cudaStream_t st) {
  return mode == 1 ? launch_t<FMT, 1>(J, sms, st) : launch_t<FMT, 0>(J, sms, st);
}

// bf16 activations -> fp16 (exact in fp16's normal range); a value outside
// it sets MOE_ERR_RANGE in the status word
__global__ void k_act_f16(const uint16_t* __restrict__ x, long n, uint16_t* __restrict__ xh,
                          int* status) {
  const long i = (long(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  if (i >= n) return;
  const uint4 v = *reinterpret_cast<const uint4*>(x + i);
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[4];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float a = __uint_as_float(in[j] << 16), b = __uint_as_float(in[j] & 0xFFFF0000u);
    bad |= !(fabsf(a) <= 65504.f) || !(fabsf(b) <= 65504.f);
    const __half2 h = __floats2half2_rn(a, b);
    out[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(xh + i) = make_uint4(out[0], out[1], out[2], out[3]);
  if (bad) atomicExch(status, int(MOE_ERR_RANGE));
}

}  // namespace

int prefill_smem(const TileGeo& g, int mode) {
  if (g.K % kPfKBlk != 0) return 0;
  // + 1024: slack to align the stages to the swizzle atom
  const int bytes = kPfRaw * raw_stage_bytes(g) + pf_stages(mode) * pf_stage_bytes(mode) + 1024;
  return bytes + int(sizeof(PfSmem)) + 1024 <= kEngineSmemMax ? bytes : 0;
}

cudaError_t launch_prefill(const PrefillJob& J, int mode, int sms, cudaStream_t st) {
  switch (J.g.fmt) {
    case MOE_FMT_AFFINE4_G64: return launch_fmt<MOE_FMT_AFFINE4_G64>(J, mode, sms, st);
    case MOE_FMT_AFFINE3_G64: return launch_fmt<MOE_FMT_AFFINE3_G64>(J, mode, sms, st);
    case MOE_FMT_W4A16_SYM_G128: return launch_fmt<MOE_FMT_W4A16_SYM_G128>(J, mode, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_act_f16(const uint16_t* x, long n, uint16_t* xh, int* status,
                           cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long threads = (n + 7) / 8;
  k_act_f16<<<unsigned((threads + 255) / 256), 256, 0, st>>>(x, n, xh, status);
  return cudaGetLastError();
}

}  // namespace moe
