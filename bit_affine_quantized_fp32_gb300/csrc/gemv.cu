// gemv.cu -- decode-path expert kernels: grouped GEMV over the selected
// experts' packed codes, the SwiGLU step, and the weighted combine.
//
// Source: "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803",
// comment "Progress on the 4-bit gate": grouped affine experts with a SwiGLU
// epilogue, decode rows summed in fp32, the slots' fma sum rounded once; and
// "Native server: --backend xpu for Nemotron on Intel Arc" (update comment):
// a row's arithmetic must not depend on which other rows share the call.
//
// Arithmetic.  For one weight row r and one 64-wide group G of the reduction:
//     sum_{i in G} (s q_i + b) x_i  =  s * (sum_{i in G} q_i x_i)  +  b * X_G
// with X_G = sum_{i in G} x_i precomputed once per operand row.  The inner sum
// runs on the tensor cores (mma.sync m16n8k16, fp32 accumulate) with the codes
// q as exact small integers in bf16/fp16 and the activations as they are, so
// every product is exact; the per-group scale and bias are applied in fp32
// registers ("dequant in registers").  W4A16 is the same with b = -8 s on the
// stored offset-binary nibble.  The down projection's operand h is fp32; it
// is split into two bf16 parts (hi + lo, 16 significant bits) that go through
// the same codes.
//
// Fragment mapping.  A warp owns a tile of 16 weight rows x 64 codes (one
// group).  Thread (g = lane/4, t = lane%4) takes the two packed words 2t and
// 2t+1 of rows g and g+8 (codes 16t..16t+15).  A word's nibble pairs (0,4),
// (1,5), (2,6), (3,7) become the MMA's k-pairs, so the operand rows (x or h)
// are stored with each 8-block permuted to [0 4 1 5 2 6 3 7]; a thread's B
// fragment for one group is then 32 contiguous bytes.
//
// Batch invariance.  Each output element is one MMA column: its value depends
// only on that token's operand row, the codes, the fixed k-order (chunks,
// groups, MMA steps) and fixed fp32 folds -- never on the other tokens, the
// bucket sizes or the number of n-tiles.
//
// Memory.  Persistent CTAs of 8 warps; each warp streams whole units
// (16 rows x one k-chunk of one expert) from HBM into its own shared-memory
// stage with 16-byte cp.async and keeps the next unit in flight.

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kGemvWarps = 8;

__host__ __device__ inline int code_bits(int fmt) {
  return fmt == MOE_FMT_AFFINE3_G64 ? 3 : 4;
}

}  // namespace

int gemv_a_pitch(int fmt, int CK) {
  const int bytes = CK * code_bits(fmt) / 8;
  return (bytes + 127) / 128 * 128 + 32;
}

int gemv_stage_bytes(int fmt, int CK) {
  const int G = fmt == MOE_FMT_W4A16_SYM_G128 ? 128 : 64;
  const int sbb = 16 * (CK / G) * 2;
  const int sb = (sbb + 15) / 16 * 16;
  return 16 * gemv_a_pitch(fmt, CK) + 2 * sb;
}

int gemv_smem_bytes(int fmt, int CK) { return kGemvWarps * 2 * gemv_stage_bytes(fmt, CK); }

namespace {

struct Geo {
  int pitch, cbytes, sbw, sbb, sbstride;
};

__device__ __forceinline__ void issue_unit(const GemvJob& J, const Geo& Q, int e, int tile, int c,
                                           uint8_t* st, int lane) {
  const size_t row0 = size_t(tile) * 16;
  const uint8_t* src = J.w + size_t(e) * J.w_estride + row0 * J.row_bytes + size_t(c) * Q.cbytes;
  const int cpr = Q.cbytes >> 4;
  for (int i = lane; i < 16 * cpr; i += kWarp) {
    const int r = i / cpr, q = i - r * cpr;
    cp_async16(st + r * Q.pitch + q * 16, src + size_t(r) * J.row_bytes + q * 16);
  }
  uint8_t* s_sm = st + 16 * Q.pitch;
  uint8_t* b_sm = s_sm + Q.sbstride;
  const int gran = J.sb_gran;
  const int gpr = Q.sbb / gran;
  const int nb = J.b ? 2 : 1;
  const size_t sb_off = size_t(e) * J.sb_estride + row0 * J.sb_cols + size_t(c) * Q.sbw;
  const uint8_t* s_src = reinterpret_cast<const uint8_t*>(J.s + sb_off);
  const uint8_t* b_src = J.b ? reinterpret_cast<const uint8_t*>(J.b + sb_off) : nullptr;
  for (int i = lane; i < nb * 16 * gpr; i += kWarp) {
    const int which = i / (16 * gpr);
    const int ii = i - which * 16 * gpr;
    const int r = ii / gpr, q = ii - r * gpr;
    const uint8_t* s = (which ? b_src : s_src) + size_t(r) * J.sb_cols * 2 + q * gran;
    uint8_t* d = (which ? b_sm : s_sm) + r * Q.sbb + q * gran;
    if (gran == 16)
      cp_async16(d, s);
    else if (gran == 8)
      cp_async8(d, s);
    else
      cp_async4(d, s);
  }
}

template <int FMT>
__device__ __forceinline__ void load_words(const uint8_t* st, const Geo& Q, int G, int g, int t,
                                           uint32_t& wr0, uint32_t& wr1, uint32_t& ws0,
                                           uint32_t& ws1) {
  if constexpr (FMT == MOE_FMT_AFFINE3_G64) {
    const int wi = G * 6 + ((3 * t) >> 1);
    const int sh = (t & 1) ? 16 : 0;
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(st + g * Q.pitch) + wi;
    const uint32_t* r1 = reinterpret_cast<const uint32_t*>(st + (g + 8) * Q.pitch) + wi;
    const uint64_t v0 = (uint64_t(r0[0]) | (uint64_t(r0[1]) << 32)) >> sh;
    const uint64_t v1 = (uint64_t(r1[0]) | (uint64_t(r1[1]) << 32)) >> sh;
    wr0 = spread3to4(uint32_t(v0) & 0xFFFFFFu);
    wr1 = spread3to4(uint32_t(v0 >> 24) & 0xFFFFFFu);
    ws0 = spread3to4(uint32_t(v1) & 0xFFFFFFu);
    ws1 = spread3to4(uint32_t(v1 >> 24) & 0xFFFFFFu);
  } else {
    const uint8_t* a = st + g * Q.pitch + G * 32 + t * 8;
    const uint2 v0 = *reinterpret_cast<const uint2*>(a);
    const uint2 v1 = *reinterpret_cast<const uint2*>(a + 8 * Q.pitch);
    wr0 = v0.x;
    wr1 = v0.y;
    ws0 = v1.x;
    ws1 = v1.y;
  }
}

template <int FMT, bool F16A, bool SPLIT, int NT>
__device__ __forceinline__ void compute_unit(const GemvJob& J, const Geo& Q, const uint8_t* st,
                                             int off, int cnt, int nt0, int tile, int c,
                                             int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int K = J.K;
  const int ksw = K >> 6;
  int brow[NT], crow0[NT], crow1[NT];
  bool bv[NT], cv0[NT], cv1[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int base = (nt0 + n) * 8;
    const int pb = base + g, p0 = base + 2 * t, p1 = p0 + 1;
    bv[n] = pb < cnt;
    cv0[n] = p0 < cnt;
    cv1[n] = p1 < cnt;
    brow[n] = bv[n] ? (J.b_row ? J.b_row[off + pb] : off + pb) : 0;
    crow0[n] = cv0[n] ? (J.b_row ? J.b_row[off + p0] : off + p0) : 0;
    crow1[n] = cv1[n] ? (J.b_row ? J.b_row[off + p1] : off + p1) : 0;
  }
  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

  const uint16_t* s_sm = reinterpret_cast<const uint16_t*>(st + 16 * Q.pitch);
  const uint16_t* b_sm = reinterpret_cast<const uint16_t*>(st + 16 * Q.pitch + Q.sbstride);
  const int ngr = J.CK >> 6;
  for (int G = 0; G < ngr; ++G) {
    const int kg = c * J.CK + G * 64;
    uint32_t wr0, wr1, ws0, ws1;
    load_words<FMT>(st, Q, G, g, t, wr0, wr1, ws0, ws1);
    uint32_t A[4][4];
    A[0][0] = codes_to_pair<F16A>(wr0);
    A[0][1] = codes_to_pair<F16A>(ws0);
    A[0][2] = codes_to_pair<F16A>(wr0 >> 4);
    A[0][3] = codes_to_pair<F16A>(ws0 >> 4);
    A[1][0] = codes_to_pair<F16A>(wr0 >> 8);
    A[1][1] = codes_to_pair<F16A>(ws0 >> 8);
    A[1][2] = codes_to_pair<F16A>(wr0 >> 12);
    A[1][3] = codes_to_pair<F16A>(ws0 >> 12);
    A[2][0] = codes_to_pair<F16A>(wr1);
    A[2][1] = codes_to_pair<F16A>(ws1);
    A[2][2] = codes_to_pair<F16A>(wr1 >> 4);
    A[2][3] = codes_to_pair<F16A>(ws1 >> 4);
    A[3][0] = codes_to_pair<F16A>(wr1 >> 8);
    A[3][1] = codes_to_pair<F16A>(ws1 >> 8);
    A[3][2] = codes_to_pair<F16A>(wr1 >> 12);
    A[3][3] = codes_to_pair<F16A>(ws1 >> 12);

    float s0, s1, b0, b1;
    if constexpr (FMT == MOE_FMT_W4A16_SYM_G128) {
      s0 = half_bits_to_float(s_sm[g * Q.sbw + (G >> 1)]);
      s1 = half_bits_to_float(s_sm[(g + 8) * Q.sbw + (G >> 1)]);
      b0 = -8.f * s0;
      b1 = -8.f * s1;
    } else {
      s0 = half_bits_to_float(s_sm[g * Q.sbw + G]);
      s1 = half_bits_to_float(s_sm[(g + 8) * Q.sbw + G]);
      b0 = half_bits_to_float(b_sm[g * Q.sbw + G]);
      b1 = half_bits_to_float(b_sm[(g + 8) * Q.sbw + G]);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      uint32_t bf[8];
      if (bv[n]) {
        const uint4* p = reinterpret_cast<const uint4*>(J.B + size_t(brow[n]) * K + kg + 16 * t);
        const uint4 x0 = __ldg(p), x1 = __ldg(p + 1);
        bf[0] = x0.x; bf[1] = x0.y; bf[2] = x0.z; bf[3] = x0.w;
        bf[4] = x1.x; bf[5] = x1.y; bf[6] = x1.z; bf[7] = x1.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) bf[i] = 0u;
      }
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int m = 0; m < 4; ++m)
        mma16816<F16A>(d, A[m][0], A[m][1], A[m][2], A[m][3], bf[2 * m], bf[2 * m + 1]);
      if constexpr (SPLIT) {
        if (bv[n]) {
          const uint4* p =
              reinterpret_cast<const uint4*>(J.Blo + size_t(brow[n]) * K + kg + 16 * t);
          const uint4 x0 = __ldg(p), x1 = __ldg(p + 1);
          bf[0] = x0.x; bf[1] = x0.y; bf[2] = x0.z; bf[3] = x0.w;
          bf[4] = x1.x; bf[5] = x1.y; bf[6] = x1.z; bf[7] = x1.w;
        }
#pragma unroll
        for (int m = 0; m < 4; ++m)
          mma16816<F16A>(d, A[m][0], A[m][1], A[m][2], A[m][3], bf[2 * m], bf[2 * m + 1]);
      }
      const float X0 = cv0[n] ? J.Bsum[size_t(crow0[n]) * ksw + (kg >> 6)] : 0.f;
      const float X1 = cv1[n] ? J.Bsum[size_t(crow1[n]) * ksw + (kg >> 6)] : 0.f;
      acc[n][0] = fmaf(s0, d[0], acc[n][0]);
      acc[n][0] = fmaf(b0, X0, acc[n][0]);
      acc[n][1] = fmaf(s0, d[1], acc[n][1]);
      acc[n][1] = fmaf(b0, X1, acc[n][1]);
      acc[n][2] = fmaf(s1, d[2], acc[n][2]);
      acc[n][2] = fmaf(b1, X0, acc[n][2]);
      acc[n][3] = fmaf(s1, d[3], acc[n][3]);
      acc[n][3] = fmaf(b1, X1, acc[n][3]);
    }
  }
  const int row = tile * 16 + g;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int base = (nt0 + n) * 8;
    const int p0 = base + 2 * t, p1 = p0 + 1;
    if (cv0[n]) {
      const int o = J.out_idx ? J.out_idx[off + p0] : off + p0;
      float* dst = J.out + (size_t(c) * J.P + o) * J.rows + row;
      dst[0] = acc[n][0];
      dst[8] = acc[n][2];
    }
    if (cv1[n]) {
      const int o = J.out_idx ? J.out_idx[off + p1] : off + p1;
      float* dst = J.out + (size_t(c) * J.P + o) * J.rows + row;
      dst[0] = acc[n][1];
      dst[8] = acc[n][3];
    }
  }
}

template <int FMT, bool F16A, bool SPLIT>
__global__ void __launch_bounds__(kGemvWarps * kWarp) k_gemv(const GemvJob J) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  Geo Q;
  Q.cbytes = J.CK * code_bits(FMT) / 8;
  Q.pitch = (Q.cbytes + 127) / 128 * 128 + 32;
  const int G = FMT == MOE_FMT_W4A16_SYM_G128 ? 128 : 64;
  Q.sbw = J.CK / G;
  Q.sbb = Q.sbw * 2;
  Q.sbstride = (16 * Q.sbb + 15) / 16 * 16;
  const int stage = 16 * Q.pitch + 2 * Q.sbstride;
  uint8_t* stages = smem + size_t(wid) * 2 * stage;

  const int n_slots = J.n_slots ? *J.n_slots : 1;
  const int tiles = J.rows >> 4;
  const int nch = J.K / J.CK;
  const int ups = tiles * nch;
  const int n_units = n_slots * ups;
  const int nw = gridDim.x * kGemvWarps;
  int u = blockIdx.x * kGemvWarps + wid;

  auto decode = [&](int uu, int& slot, int& tile, int& c) {
    slot = uu / ups;
    const int rem = uu - slot * ups;
    tile = rem / nch;
    c = rem - tile * nch;
  };
  auto slot_expert = [&](int slot) { return J.n_slots ? J.slot_expert[slot] : J.fixed_expert; };

  if (u < n_units) {
    int slot, tile, c;
    decode(u, slot, tile, c);
    issue_unit(J, Q, slot_expert(slot), tile, c, stages, lane);
  }
  cp_async_commit();
  for (int it = 0; u < n_units; ++it, u += nw) {
    const int un = u + nw;
    if (un < n_units) {
      int slot, tile, c;
      decode(un, slot, tile, c);
      issue_unit(J, Q, slot_expert(slot), tile, c, stages + ((it + 1) & 1) * stage, lane);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncwarp();
    int slot, tile, c;
    decode(u, slot, tile, c);
    const int off = J.n_slots ? J.slot_off[slot] : 0;
    const int cnt = J.n_slots ? J.slot_cnt[slot] : J.fixed_cnt;
    const uint8_t* st = stages + (it & 1) * stage;
    const int ntiles = (cnt + 7) >> 3;
    for (int nt0 = 0; nt0 < ntiles; nt0 += 4) {
      const int nn = min(4, ntiles - nt0);
      if (nn == 4)
        compute_unit<FMT, F16A, SPLIT, 4>(J, Q, st, off, cnt, nt0, tile, c, lane);
      else if (nn == 3)
        compute_unit<FMT, F16A, SPLIT, 3>(J, Q, st, off, cnt, nt0, tile, c, lane);
      else if (nn == 2)
        compute_unit<FMT, F16A, SPLIT, 2>(J, Q, st, off, cnt, nt0, tile, c, lane);
      else
        compute_unit<FMT, F16A, SPLIT, 1>(J, Q, st, off, cnt, nt0, tile, c, lane);
    }
    __syncwarp();
  }
  cp_async_wait<0>();
}

// h = silu(sum_c gate) * (sum_c up), split into bf16 hi/lo, k-permuted, with
// per-64-group sums of (hi + lo).  One warp per (position, 64-group).
__global__ void k_hprep(const float* __restrict__ part, int nch, int P, int I,
                        uint16_t* __restrict__ hh, uint16_t* __restrict__ hl,
                        float* __restrict__ hsum, float* __restrict__ hout) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int ng = I >> 6;
  if (gw >= P * ng) return;
  const int p = gw / ng, G = gw - p * ng;
  const int j0 = G * 64 + 2 * lane;
  float a0 = 0.f, a1 = 0.f, u0 = 0.f, u1 = 0.f;
  for (int c = 0; c < nch; ++c) {
    const float* pr = part + (size_t(c) * P + p) * 2 * I;
    const float2 av = *reinterpret_cast<const float2*>(pr + j0);
    const float2 uv = *reinterpret_cast<const float2*>(pr + I + j0);
    a0 += av.x;
    a1 += av.y;
    u0 += uv.x;
    u1 += uv.y;
  }
  const float h0 = a0 / (1.f + expf(-a0)) * u0;
  const float h1 = a1 / (1.f + expf(-a1)) * u1;
  const __nv_bfloat16 hi0 = __float2bfloat16_rn(h0), hi1 = __float2bfloat16_rn(h1);
  const __nv_bfloat16 lo0 = __float2bfloat16_rn(h0 - __bfloat162float(hi0));
  const __nv_bfloat16 lo1 = __float2bfloat16_rn(h1 - __bfloat162float(hi1));
  const size_t rb = size_t(p) * I;
  hh[rb + kperm_pos(j0)] = __bfloat16_as_ushort(hi0);
  hh[rb + kperm_pos(j0 + 1)] = __bfloat16_as_ushort(hi1);
  hl[rb + kperm_pos(j0)] = __bfloat16_as_ushort(lo0);
  hl[rb + kperm_pos(j0 + 1)] = __bfloat16_as_ushort(lo1);
  if (hout) {
    hout[rb + j0] = h0;
    hout[rb + j0 + 1] = h1;
  }
  float s = (__bfloat162float(hi0) + __bfloat162float(lo0)) +
            (__bfloat162float(hi1) + __bfloat162float(lo1));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) hsum[size_t(p) * ng + G] = s;
}

// x rows -> k-permuted copy + per-64-group fp32 sums.  One warp per (t, group).
__global__ void k_xprep(const uint16_t* __restrict__ x, int T, int H, int f16,
                        uint16_t* __restrict__ xperm, float* __restrict__ xsum) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int ng = H >> 6;
  if (gw >= T * ng) return;
  const int t = gw / ng, G = gw - t * ng;
  const int j0 = G * 64 + 2 * lane;
  const size_t rb = size_t(t) * H;
  const uint32_t v = *reinterpret_cast<const uint32_t*>(x + rb + j0);
  const uint16_t v0 = uint16_t(v & 0xFFFFu), v1 = uint16_t(v >> 16);
  xperm[rb + kperm_pos(j0)] = v0;
  xperm[rb + kperm_pos(j0 + 1)] = v1;
  float s = act_to_float(v0, f16) + act_to_float(v1, f16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) xsum[size_t(t) * ng + G] = s;
}

// out[t, h] = round( sum_j w[t, j] * y[t*k + j, h]  (+ s_t * ysh[t, h]) )
__global__ void k_combine(const float* __restrict__ y, const float* __restrict__ w, int k,
                          const float* __restrict__ ysh, const float* __restrict__ sg, int T,
                          int H, int f16, uint16_t* __restrict__ out) {
  const size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= size_t(T) * H) return;
  const int t = int(i / H);
  const int h = int(i - size_t(t) * H);
  float acc = 0.f;
  for (int j = 0; j < k; ++j) acc = fmaf(w[t * k + j], y[(size_t(t) * k + j) * H + h], acc);
  if (ysh) acc = fmaf(sg ? sg[t] : 1.f, ysh[size_t(t) * H + h], acc);
  out[i] = float_to_act_bits(acc, f16 != 0);
}

template <int FMT, bool F16A, bool SPLIT>
cudaError_t launch_gemv_t(const GemvJob& J, int sms, cudaStream_t st) {
  const int smem = gemv_smem_bytes(FMT, J.CK);
  static unsigned long long configured = 0;  // one bit per device, per template instance
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    e = cudaFuncSetAttribute(k_gemv<FMT, F16A, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             200 * 1024);
    if (e != cudaSuccess) return e;
    configured |= bit;
  }
  const int warps_needed = J.max_units;
  int blocks = (warps_needed + kGemvWarps - 1) / kGemvWarps;
  const int per_sm = smem > 110 * 1024 ? 1 : 2;
  blocks = blocks < sms * per_sm ? blocks : sms * per_sm;
  if (blocks < 1) blocks = 1;
  k_gemv<FMT, F16A, SPLIT><<<blocks, kGemvWarps * kWarp, smem, st>>>(J);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const GemvJob& J, bool f16a, bool split, int sms, cudaStream_t st) {
  switch (J.fmt) {
    case MOE_FMT_AFFINE4_G64:
      if (split) return launch_gemv_t<MOE_FMT_AFFINE4_G64, false, true>(J, sms, st);
      return f16a ? launch_gemv_t<MOE_FMT_AFFINE4_G64, true, false>(J, sms, st)
                  : launch_gemv_t<MOE_FMT_AFFINE4_G64, false, false>(J, sms, st);
    case MOE_FMT_AFFINE3_G64:
      if (split) return launch_gemv_t<MOE_FMT_AFFINE3_G64, false, true>(J, sms, st);
      return f16a ? launch_gemv_t<MOE_FMT_AFFINE3_G64, true, false>(J, sms, st)
                  : launch_gemv_t<MOE_FMT_AFFINE3_G64, false, false>(J, sms, st);
    case MOE_FMT_W4A16_SYM_G128:
      if (split) return launch_gemv_t<MOE_FMT_W4A16_SYM_G128, false, true>(J, sms, st);
      return f16a ? launch_gemv_t<MOE_FMT_W4A16_SYM_G128, true, false>(J, sms, st)
                  : launch_gemv_t<MOE_FMT_W4A16_SYM_G128, false, false>(J, sms, st);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_hprep(const float* part, int nch, int P, int I, uint16_t* hh, uint16_t* hl,
                         float* hsum, float* hout, cudaStream_t st) {
  const long warps = long(P) * (I / 64);
  if (warps == 0) return cudaSuccess;
  const int blocks = int((warps + 7) / 8);
  k_hprep<<<blocks, 256, 0, st>>>(part, nch, P, I, hh, hl, hsum, hout);
  return cudaGetLastError();
}

cudaError_t launch_xprep(const uint16_t* x, int T, int H, bool f16, uint16_t* xperm, float* xsum,
                         cudaStream_t st) {
  const long warps = long(T) * (H / 64);
  if (warps == 0) return cudaSuccess;
  const int blocks = int((warps + 7) / 8);
  k_xprep<<<blocks, 256, 0, st>>>(x, T, H, f16 ? 1 : 0, xperm, xsum);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* y, const float* w, int k, const float* ysh,
                           const float* sg, int T, int H, bool f16, uint16_t* out,
                           cudaStream_t st) {
  const size_t n = size_t(T) * H;
  if (n == 0) return cudaSuccess;
  const int blocks = int((n + 255) / 256);
  k_combine<<<blocks, 256, 0, st>>>(y, w, k, ysh, sg, T, H, f16 ? 1 : 0, out);
  return cudaGetLastError();
}

}  // namespace moe
