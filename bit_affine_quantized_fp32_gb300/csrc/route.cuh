// route.cuh -- routing as CTA/warp-level device functions: router logits,
// top-k with routing weights, bucketing, active-expert slots.  Used by the
// standalone routing kernels and by the fused decode kernel.
//
// Source: "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803",
// comment "Progress on the 4-bit gate": fp32 logits over the experts and the
// shared expert's gate row, top-k by logit with ties to the lower id, weights
// exp(l - l_top) over the k (normalised over the k here), the shared expert
// weighted by sigmoid(gate).  Bucketing (a stable counting sort of the
// assignments by expert) feeds the grouped experts of "Sage-A1.5 ... on the
// XPU backend #1329" (Proposal: grouped MoE).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kRouterTT = 64;  // tokens per pass of a router block

// Four consecutive weights of row r at column k (k % 4 == 0) as fp32.
__device__ __forceinline__ void router_load_w4(int fmt, const void* q, const uint16_t* s,
                                               const uint16_t* b, int r, int H, int k,
                                               float (&w)[4], bool rb) {
  if (fmt == MOE_FMT_F32) {
    const float4 v =
        *reinterpret_cast<const float4*>(static_cast<const float*>(q) + size_t(r) * H + k);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if (fmt == MOE_FMT_BF16 || fmt == MOE_FMT_F16) {
    const uint2 v =
        *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(q) + size_t(r) * H + k);
    const bool f16 = fmt == MOE_FMT_F16;
    w[0] = act_to_float(uint16_t(v.x & 0xFFFF), f16);
    w[1] = act_to_float(uint16_t(v.x >> 16), f16);
    w[2] = act_to_float(uint16_t(v.y & 0xFFFF), f16);
    w[3] = act_to_float(uint16_t(v.y >> 16), f16);
  } else {  // MOE_FMT_AFFINE8_G64: w = scale * q + bias
    const uint32_t word = static_cast<const uint32_t*>(q)[size_t(r) * (H / 4) + k / 4];
    const size_t gi = size_t(r) * (H / 64) + k / 64;
    const float sc = half_bits_to_float(s[gi]);
    const float bi = half_bits_to_float(b[gi]);
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = fmaf(sc, float((word >> (8 * j)) & 0xFFu), bi);
  }
  if (rb) {  // the engine's bf16 rounding chain: rows stored as bf16
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = round_bf16(w[j]);
  }
}

// One warp's share of the router: the dot products of router row `row` (the
// shared-gate row when row == E) over k-split q of KS (4*NI columns per lane,
// held in registers) with tokens 0..tn-1 of xs (row stride H; global or
// shared memory).  Lane order and xor tree are fixed; lane 0 writes token
// t's partial sum to out[t * ostride].  pre() runs between the weight loads
// and the first read of xs (the fused kernel waits for its x copy there).
struct NoPre {
  __device__ void operator()() const {}
};

template <int NI, class Pre>
__device__ __forceinline__ void router_warp(const RouterJob& J, int KS, int row, int q,
                                            const uint16_t* xs, int tn, float* out, int ostride,
                                            const Pre& pre) {
  const int lane = threadIdx.x & 31;
  const int kq = q * (J.H / KS);
  float w[NI][4];
  const bool gate = row >= J.E;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int k = kq + 128 * i + 4 * lane;
    if (gate)
      router_load_w4(J.gfmt, J.gq, J.gs, J.gb, 0, J.H, k, w[i], J.round_bf16 != 0);
    else
      router_load_w4(J.fmt, J.q, J.s, J.b, row, J.H, k, w[i], J.round_bf16 != 0);
  }
  pre();
  // 8 tokens per pass: every x load of a pass is issued before its sums (a
  // token past the end re-reads the last row; its sum is not written)
  for (int tl = 0; tl < tn; tl += 8) {
    uint2 xv[8][NI];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint16_t* xr = xs + size_t(min(tl + u, tn - 1)) * J.H + kq + 4 * lane;
#pragma unroll
      for (int i = 0; i < NI; ++i) xv[u][i] = *reinterpret_cast<const uint2*>(xr + 128 * i);
    }
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      acc[u] = 0.f;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const uint2 v = xv[u][i];
        acc[u] = fmaf(w[i][0], act_to_float(uint16_t(v.x & 0xFFFF), J.f16), acc[u]);
        acc[u] = fmaf(w[i][1], act_to_float(uint16_t(v.x >> 16), J.f16), acc[u]);
        acc[u] = fmaf(w[i][2], act_to_float(uint16_t(v.y & 0xFFFF), J.f16), acc[u]);
        acc[u] = fmaf(w[i][3], act_to_float(uint16_t(v.y >> 16), J.f16), acc[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
      if (lane == 0 && tl + u < tn) out[size_t(tl + u) * ostride] = acc[u];
    }
  }
}

template <class Pre = NoPre>
__device__ __forceinline__ void router_warp_any(const RouterJob& J, int KS, int row, int q,
                                                const uint16_t* xs, int tn, float* out,
                                                int ostride, const Pre& pre = Pre()) {
  const int NI_ = J.H / (KS * 128);
  if (NI_ == 1)
    router_warp<1>(J, KS, row, q, xs, tn, out, ostride, pre);
  else if (NI_ == 2)
    router_warp<2>(J, KS, row, q, xs, tn, out, ostride, pre);
  else if (NI_ == 3)
    router_warp<3>(J, KS, row, q, xs, tn, out, ostride, pre);
  else
    router_warp<4>(J, KS, row, q, xs, tn, out, ostride, pre);
}

// A logit from its KS partial sums (stride apart), added in split order, plus
// the row's bias.
__device__ __forceinline__ float router_finalize(const float* p, size_t stride, int KS,
                                                 const float* bias) {
  float s = 0.f;
  for (int q = 0; q < KS; ++q) s += p[q * stride];
  if (bias) s += *bias;
  return s;
}


// Split q of R consecutive router rows row0.. (rows >= nrows skipped; the
// shared-gate row is row E) for all T tokens of J.x, by one warp: every
// weight of the split in registers, then for each pass of 8 tokens the x
// values loaded once and used for all R rows.  Per (row, token) the sum has
// the lane order and xor tree of router_warp, so the partials are the same
// bits.  Lane 0 writes part[(r * KS + q) * T + t].
template <int NI, int R>
__device__ __forceinline__ void router_warp_rows(const RouterJob& J, int KS, int row0, int nrows,
                                                 int q, float* part, const uint16_t* xs = nullptr,
                                                 int tn = -1) {
  const int lane = threadIdx.x & 31;
  const int kq = q * (J.H / KS);
  const int T = tn < 0 ? J.T : tn;
  if (!xs) xs = J.x;
  float w[R][NI][4];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int row = row0 + r < nrows ? row0 + r : row0;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int k = kq + 128 * i + 4 * lane;
      if (row >= J.E)
        router_load_w4(J.gfmt, J.gq, J.gs, J.gb, 0, J.H, k, w[r][i], J.round_bf16 != 0);
      else
        router_load_w4(J.fmt, J.q, J.s, J.b, row, J.H, k, w[r][i], J.round_bf16 != 0);
    }
  }
  for (int tl = 0; tl < T; tl += 8) {
    uint2 xv[8][NI];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint16_t* xr = xs + size_t(min(tl + u, T - 1)) * J.H + kq + 4 * lane;
#pragma unroll
      for (int i = 0; i < NI; ++i) xv[u][i] = *reinterpret_cast<const uint2*>(xr + 128 * i);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float acc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc[u] = 0.f;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const uint2 v = xv[u][i];
          acc[u] = fmaf(w[r][i][0], act_to_float(uint16_t(v.x & 0xFFFF), J.f16), acc[u]);
          acc[u] = fmaf(w[r][i][1], act_to_float(uint16_t(v.x >> 16), J.f16), acc[u]);
          acc[u] = fmaf(w[r][i][2], act_to_float(uint16_t(v.y & 0xFFFF), J.f16), acc[u]);
          acc[u] = fmaf(w[r][i][3], act_to_float(uint16_t(v.y >> 16), J.f16), acc[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
        if (lane == 0 && tl + u < T && row0 + r < nrows)
          part[size_t(r * KS + q) * T + tl + u] = acc[u];
      }
    }
  }
}

// Rows two at a time when a warp's split is at most 2 x 128 columns (the
// weights of both rows stay in registers), else one at a time.
__device__ __forceinline__ void router_warp_rows_any(const RouterJob& J, int KS, int row0,
                                                     int R, int nrows, int q, float* part) {
  const int NI_ = J.H / (KS * 128);
  for (int r0 = 0; r0 < R;) {
    float* pr = part + size_t(r0) * KS * J.T;
    if (NI_ <= 2 && R - r0 >= 2) {
      if (NI_ == 1)
        router_warp_rows<1, 2>(J, KS, row0 + r0, nrows, q, pr);
      else
        router_warp_rows<2, 2>(J, KS, row0 + r0, nrows, q, pr);
      r0 += 2;
    } else {
      if (NI_ == 1)
        router_warp_rows<1, 1>(J, KS, row0 + r0, nrows, q, pr);
      else if (NI_ == 2)
        router_warp_rows<2, 1>(J, KS, row0 + r0, nrows, q, pr);
      else if (NI_ == 3)
        router_warp_rows<3, 1>(J, KS, row0 + r0, nrows, q, pr);
      else
        router_warp_rows<4, 1>(J, KS, row0 + r0, nrows, q, pr);
      r0 += 1;
    }
  }
}

// Router block of the standalone kernel: rows [rb * R, rb * R + R) (the
// shared-gate row is row E) for tokens [t0, t0 + tn), tn <= kRouterTT, with
// warp q computing split q of all R rows (x loaded once per warp for the R
// rows) into part [R * KS][kRouterTT], then every (row, token) finalised in
// split order.  The same per-(row, token) arithmetic as router_warp, so the
// same bits as the fused kernel's router.  Needs blockDim.x == 32 * KS.
template <int R>
__device__ __forceinline__ void router_block_rows(const RouterJob& J, int KS, int rb, float* part,
                                                  int t0, int tn) {
  const int wid = threadIdx.x >> 5;
  const int nrows = J.E + (J.gq ? 1 : 0);
  const int row0 = rb * R;
  const int NI_ = J.H / (KS * 128);
  const uint16_t* xs = J.x + size_t(t0) * J.H;
  if (NI_ == 1)
    router_warp_rows<1, R>(J, KS, row0, nrows, wid, part, xs, tn);
  else if (NI_ == 2)
    router_warp_rows<2, R>(J, KS, row0, nrows, wid, part, xs, tn);
  else
    for (int r = 0; r < R; ++r) {  // wide splits: one row at a time
      if (NI_ == 3)
        router_warp_rows<3, 1>(J, KS, row0 + r, nrows, wid, part + size_t(r) * KS * tn, xs, tn);
      else
        router_warp_rows<4, 1>(J, KS, row0 + r, nrows, wid, part + size_t(r) * KS * tn, xs, tn);
    }
  __syncthreads();
  for (int i = threadIdx.x; i < R * tn; i += blockDim.x) {
    const int r2 = i / tn, tl = i - r2 * tn;
    const int row2 = row0 + r2;
    if (row2 >= nrows) continue;
    const float* p = part + (r2 * KS) * tn + tl;
    if (row2 < J.E)
      J.logits[size_t(t0 + tl) * J.E + row2] =
          router_finalize(p, tn, KS, J.bias ? J.bias + row2 : nullptr);
    else
      J.gate_logit[t0 + tl] = router_finalize(p, tn, KS, nullptr);
  }
  __syncthreads();
}

// The fused kernel's router block rb: rows [rb*RPB, rb*RPB + RPB) (the
// shared-gate row is row E), warp (r, q) computing split q of row r into
// part [RPB * KS][T] (shared; RPB * KS * T <= 512 floats), then every
// (row, token) finalised in split order (router_finalize, as
// router_block_rows does).  Threads 0..511 (the consumer warps) call it; it synchronises them
// with named barrier 2 only, so the CTA's other warps go on meanwhile.
// With `tagged` set, each logit (and the shared-gate logit, row E) is
// published instead as one 64-bit word tagged[t * TS + row] = gen << 32 |
// bits(logit): a reader that sees the call's generation number sees the
// final value, so no fence or counter is needed.
__device__ __forceinline__ void router_rows_cta(const RouterJob& J, int KS, int RPB, int rb,
                                                float* part, unsigned long long* tagged = nullptr,
                                                int TS = 0, unsigned gen = 0) {
  const int wid = threadIdx.x >> 5;
  const int nrows = J.E + (J.gq ? 1 : 0);
  const int row0 = rb * RPB;
  // the bias of this thread's first finalisation, fetched before the sums
  float bias0 = 0.f;
  if (J.bias && int(threadIdx.x) < RPB * J.T) {
    const int row2 = row0 + int(threadIdx.x) / J.T;
    if (row2 < J.E) bias0 = J.bias[row2];
  }
  // warp (r, q) computes split q of row row0 + r: one row per warp keeps the
  // dependent chains short (x is read through L2 once per row)
  if (wid < RPB * KS) {
    const int r = wid / KS, q = wid - r * KS;
    router_warp_rows_any(J, KS, row0 + r, 1, nrows, q, part + size_t(r) * KS * J.T);
  }
  asm volatile("bar.sync 2, 512;\n" ::: "memory");
  for (int i = threadIdx.x; i < RPB * J.T; i += 512) {
    const int r2 = i / J.T, tl = i - r2 * J.T;
    const int row2 = row0 + r2;
    if (row2 >= nrows) continue;
    const float* p = part + (r2 * KS) * J.T + tl;
    const float v =
        row2 < J.E ? router_finalize(p, J.T, KS,
                                     J.bias ? (i == int(threadIdx.x) ? &bias0 : J.bias + row2)
                                            : nullptr)
                   : router_finalize(p, J.T, KS, nullptr);
    if (tagged)
      st_relaxed_u64(tagged + size_t(tl) * TS + row2,
                     (static_cast<unsigned long long>(gen) << 32) | __float_as_uint(v));
    else if (row2 < J.E)
      J.logits[size_t(tl) * J.E + row2] = v;
    else
      J.gate_logit[tl] = v;
  }
  asm volatile("bar.sync 2, 512;\n" ::: "memory");
}

// Ranking key of (logit v, expert id): a larger key ranks first.  The high
// word is an order-preserving image of the float (-0 folded onto +0, so equal
// logits tie), 0 for NaN; the low word is 256 - id, so equal logits go to the
// lower id and every real key is >= 1 (0 marks "no expert").
__device__ __forceinline__ unsigned long long rank_key(float v, int id) {
  unsigned u = __float_as_uint(v == 0.f ? 0.f : v);
  unsigned hi = (v != v) ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
  return ((unsigned long long)hi << 32) | unsigned(256 - id);
}

__device__ __forceinline__ float key_value(unsigned hi) {
  if (hi == 0u) return __uint_as_float(0x7fc00000u);
  return __uint_as_float((hi & 0x80000000u) ? (hi & 0x7fffffffu) : ~hi);
}

// Selection of the top k of token t from each lane's keys (8 per lane, any
// experts; see rank_key): each lane sorts its keys once; each of the k rounds
// takes the warp maximum of the lanes' heads (redux.max on the high word, and
// on the low word only when several lanes tie) and the winning lane pops its
// head.  Then w_j = exp(l_j - l_0) / sum over the k, the exponentials by lanes
// 0..k-1 in parallel and the sum in slot order.  Lanes 0..k-1 write
// idx/w[t*k + j] (and idx2/w2 when given); lane 0 writes sg[t] from the gate
// logit gl when has_gate.  rb (the engine's bf16 rounding chain): each slot
// weight is stored as bf16(w) and the shared weight as bf16(sigmoid(bf16(gl))).
__device__ __forceinline__ void topk_select(unsigned long long (&key)[8], int t, int k,
                                            int32_t* idx, float* w, float* sg, bool has_gate,
                                            float gl, int32_t* idx2, float* w2, bool rb) {
  const int lane = threadIdx.x & 31;
  // sorting network (descending), 19 compare-exchanges
#define MOE_CX(a, b)                                  \
  {                                                   \
    const unsigned long long x_ = key[a], y_ = key[b]; \
    key[a] = x_ > y_ ? x_ : y_;                       \
    key[b] = x_ > y_ ? y_ : x_;                       \
  }
  MOE_CX(0, 1) MOE_CX(2, 3) MOE_CX(4, 5) MOE_CX(6, 7)
  MOE_CX(0, 2) MOE_CX(1, 3) MOE_CX(4, 6) MOE_CX(5, 7)
  MOE_CX(1, 2) MOE_CX(5, 6) MOE_CX(0, 4) MOE_CX(3, 7)
  MOE_CX(1, 5) MOE_CX(2, 6)
  MOE_CX(1, 4) MOE_CX(3, 6)
  MOE_CX(2, 4) MOE_CX(3, 5)
  MOE_CX(3, 4)
#undef MOE_CX
  int my_e = 0;
  float my_v = 0.f, top = 0.f;
  // rounds as a rolled loop: this code runs once per call, so a small
  // footprint matters more than the loop overhead
#pragma unroll 1
  for (int r = 0; r < 8; ++r) {
    if (r < k) {
      const unsigned hi = unsigned(key[0] >> 32), lo = unsigned(key[0]);
      const unsigned mh = __reduce_max_sync(0xffffffffu, hi);
      const unsigned tie = __ballot_sync(0xffffffffu, hi == mh);
      const unsigned ml =
          (tie & (tie - 1u)) ? __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u)
                             : __shfl_sync(0xffffffffu, lo, __ffs(tie) - 1);
      if (hi == mh && lo == ml) {
#pragma unroll
        for (int i = 0; i < 7; ++i) key[i] = key[i + 1];
        key[7] = 0ull;
      }
      const float v = key_value(mh);
      if (r == 0) top = v;
      if (lane == r) {
        my_e = 256 - int(ml);
        my_v = v;
      }
    }
  }
  const float ex = lane < k ? expf(my_v - top) : 0.f;
  float den = 0.f;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const float er = __shfl_sync(0xffffffffu, ex, r);
    if (r < k) den += er;
  }
  if (lane < k) {
    const float wr = rb ? round_bf16(ex / den) : ex / den;
    idx[size_t(t) * k + lane] = my_e;
    w[size_t(t) * k + lane] = wr;
    if (idx2) idx2[size_t(t) * k + lane] = my_e;
    if (w2) w2[size_t(t) * k + lane] = wr;
  }
  if (lane == 0 && has_gate && sg)
    sg[t] = rb ? round_bf16(1.f / (1.f + expf(-round_bf16(gl)))) : 1.f / (1.f + expf(-gl));
}

// Top-k + weights of token t by one warp from fp32 logits [T][E] (E <= 256),
// lane l taking experts 8l..8l+7, read from shared memory (SMEM) or through
// L2 (they may have been written by other CTAs).
template <bool SMEM = false>
__device__ __forceinline__ void topk_warp(const float* logits, const float* gate_logit, int t,
                                          int E, int k, int32_t* idx, float* w, float* sg,
                                          int32_t* idx2, float* w2, bool rb) {
  const int lane = threadIdx.x & 31;
  const float* row = logits + size_t(t) * E;
  float v[8];
  if ((E & 7) == 0 && 8 * lane < E && ((reinterpret_cast<uintptr_t>(row) & 15u) == 0)) {
    const float4 a = SMEM ? *reinterpret_cast<const float4*>(row + 8 * lane)
                          : __ldcg(reinterpret_cast<const float4*>(row + 8 * lane));
    const float4 b = SMEM ? *reinterpret_cast<const float4*>(row + 8 * lane + 4)
                          : __ldcg(reinterpret_cast<const float4*>(row + 8 * lane + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = 8 * lane + i;
      v[i] = e < E ? (SMEM ? row[e] : __ldcg(row + e)) : 0.f;
    }
  }
  unsigned long long key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * lane + i;
    key[i] = e < E ? rank_key(v[i], e) : 0ull;
  }
  float gl = 0.f;
  if (gate_logit) gl = SMEM ? gate_logit[t] : __ldcg(gate_logit + t);
  topk_select(key, t, k, idx, w, sg, gate_logit != nullptr, gl, idx2, w2, rb);
}

// topk_warp on logits published as tagged words (router_rows_cta): the warp
// polls token t's row until every word carries generation `gen`, bounded by
// the CTA's wait limit (on a timeout it records MOE_ERR_TIMEOUT and goes on
// with whatever it read).  Row stride TS (even), the shared-gate logit at
// column E when has_gate.
__device__ __forceinline__ void topk_warp_tagged(const unsigned long long* tagged, int TS,
                                                 unsigned gen, bool has_gate, int t, int E, int k,
                                                 int32_t* idx, float* w, float* sg, int32_t* idx2,
                                                 float* w2, bool rb, WaitCtl* wc, int* status) {
  const int lane = threadIdx.x & 31;
  const unsigned long long* row = tagged + size_t(t) * TS;
  float v[8];
  float gl = 0.f;
  const unsigned long long t0 = global_ns();
  for (;;) {
    bool ok = true;
    if (8 * lane + 8 <= E) {
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        unsigned long long a, b;
        ld_relaxed_v2u64(row + 8 * lane + i, a, b);
        ok = ok && unsigned(a >> 32) == gen && unsigned(b >> 32) == gen;
        v[i] = __uint_as_float(unsigned(a));
        v[i + 1] = __uint_as_float(unsigned(b));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[i] = 0.f;
        if (8 * lane + i < E) {
          const unsigned long long a = ld_relaxed_u64(row + 8 * lane + i);
          ok = ok && unsigned(a >> 32) == gen;
          v[i] = __uint_as_float(unsigned(a));
        }
      }
    }
    if (has_gate && lane == 0) {
      const unsigned long long a = ld_relaxed_u64(row + E);
      ok = ok && unsigned(a >> 32) == gen;
      gl = __uint_as_float(unsigned(a));
    }
    if (__all_sync(0xffffffffu, ok)) break;
    if (*(volatile int*)&wc->skip) break;
    __nanosleep(100);  // every CTA polls the same lines: keep L2 free for the writers
    if (global_ns() - t0 > wc->limit_ns) {
      if (lane == 0) {
        wc->skip = 1;
        atomicExch(status, int(MOE_ERR_TIMEOUT));
      }
      break;
    }
  }
  unsigned long long key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * lane + i;
    key[i] = e < E ? rank_key(v[i], e) : 0ull;
  }
  topk_select(key, t, k, idx, w, sg, has_gate, gl, idx2, w2, rb);
}

// Shared memory of bucket_cta (up to 32 warps, up to 256 experts).
struct BucketSmem {
  int wc[32][256];  // per-warp counts, then per-warp cursors
  int base[256];    // first bucket position of each expert
  int wsum[8];
};

// Stable counting sort of the N assignment ids by expert (one CTA of 32
// warps): warp w owns a contiguous range of assignments, taken in rounds of
// 32 in order.  Pass 1 counts each expert per warp (warp match: one add per
// expert and round), then every expert's counts are prefix-summed over the
// warps and its total over the experts (the bucket offsets), and pass 2 puts
// each assignment at base[e] + (earlier assignments of e in earlier warps and
// rounds) + (its rank among this round's lanes with expert e).  Ids outside
// 0..E-1 are skipped.
__device__ __forceinline__ void bucket_cta(const int32_t* idx, int N, int E, int32_t* offsets,
                                           int32_t* perm, BucketSmem& S) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int NW = blockDim.x >> 5;
  const int C = (((N + NW - 1) / NW) + 31) & ~31;  // assignments per warp
  const int a0 = min(N, wid * C), a1 = min(N, a0 + C);
  for (int i = lane; i < 256; i += 32) S.wc[wid][i] = 0;
  __syncwarp();
  for (int b = a0; b < a1; b += 32) {
    const int a = b + lane;
    int e = a < a1 ? __ldcg(idx + a) : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (__ffs(peers) - 1) == lane) S.wc[wid][e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // thread e: exclusive prefix of expert e's counts over the warps (in place)
  int tot = 0;
  if (tid < 256) {
    for (int w = 0; w < NW; ++w) {
      const int c = S.wc[w][tid];
      S.wc[w][tid] = tot;
      tot += c;
    }
    if (tid >= E) tot = 0;
  }
  // exclusive scan of the totals over the experts (the first 8 warps)
  int incl = tot;
  if (tid < 256) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) S.wsum[wid] = incl;
  }
  __syncthreads();
  if (tid < 256) {
    int pre = 0;
    for (int i = 0; i < wid; ++i) pre += S.wsum[i];
    incl += pre;
    S.base[tid] = incl - tot;
    if (tid < E) offsets[tid + 1] = incl;
    if (tid == 0) offsets[0] = 0;
  }
  __syncthreads();
  for (int b = a0; b < a1; b += 32) {
    const int a = b + lane;
    int e = a < a1 ? __ldcg(idx + a) : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) perm[S.base[e] + S.wc[wid][e] + __popc(peers & ((1u << lane) - 1u))] = a;
    __syncwarp();
    if (e >= 0 && (__ffs(peers) - 1) == lane) S.wc[wid][e] += __popc(peers);
    __syncwarp();
  }
}

// Sub-slots from the bucket offsets: every active expert (ascending id) with
// more than cmin and at most cmax assignments is cut into runs of at most
// `run` bucket positions (8 for the decode units, the N tile for the prefill
// GEMMs).  Needs blockDim.x >= 256 (the first 256 threads scan).
__device__ __forceinline__ void subslots_cta(const int32_t* offsets, int E, int* nss, int* se,
                                             int* so, int* sc, int* wcount /* 8 ints of smem */,
                                             int run = 8, int cmin = 0, int cmax = 1 << 30) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int c = 0, off = 0, nsub = 0, incl = 0;
  if (tid < 256) {
    if (tid < E) {
      off = __ldcg(offsets + tid);
      c = __ldcg(offsets + tid + 1) - off;
      if (c <= cmin || c > cmax) c = 0;
    }
    nsub = (c + run - 1) / run;
    incl = nsub;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wcount[wid] = incl;
  }
  __syncthreads();
  if (tid < 256) {
    int pre = 0;
    for (int i = 0; i < wid; ++i) pre += wcount[i];
    const int base = pre + incl - nsub;
    for (int i = 0; i < nsub; ++i) {
      se[base + i] = tid;
      so[base + i] = off + run * i;
      sc[base + i] = min(run, c - run * i);
    }
    if (tid == 0) {
      int tot = 0;
      for (int i = 0; i < 8; ++i) tot += wcount[i];
      *nss = tot;
    }
  }
  __syncthreads();
}

// Routing of a decode batch (T <= 32, T*k <= 256 assignments) by one CTA,
// every result in shared memory: top-k + weights per token (topk_warp), the
// stable counting
// sort of the assignments by expert (as bucket_cta) and the sub-slot table
// (as subslots_cta).  Same definitions as the standalone kernels, same bits.
constexpr int kMaxSubFused = 296;  // sub-slots of a call with T*k <= 256

struct RouteTable {
  int idx[256];                // [T*k] experts by slot
  float w[256];                // [T*k] routing weights
  float sg[32];                // [T] shared-gate weights
  int perm[256];               // bucket position -> assignment id
  int ss_e[kMaxSubFused];      // sub-slot -> expert
  int ss_off[kMaxSubFused];    //            first bucket position
  int ss_cnt[kMaxSubFused];    //            tokens (1..8)
  int nss;
  int cnt[256];                // scratch
  int off[256];
  int sbase[256];
  int wsum[8];
  int wsub[8];
};

// logits [T][E] and gate_logit [T] (nullable) written by other CTAs; wc:
// 8*256 ints of shared scratch.  user_idx/user_w (nullable) receive the top-k
// outputs.  All threads of the CTA call it (blockDim.x >= 256).
// With `tagged` set, the logits come from tagged words of generation gen
// (row stride TS) instead, polled until they are all published.
__device__ __forceinline__ void route_table_cta(const float* logits, const float* gate_logit,
                                                int T, int E, int k, int32_t* user_idx,
                                                float* user_w, int (*wc)[256], RouteTable& S,
                                                bool rb, const unsigned long long* tagged = nullptr,
                                                int TS = 0, unsigned gen = 0,
                                                bool has_gate = false, WaitCtl* wctl = nullptr,
                                                int* status = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int NT = blockDim.x, NW = NT >> 5;
  for (int i = tid; i < 256; i += NT) S.cnt[i] = 0;
  for (int i = tid; i < 8 * 256; i += NT) wc[i >> 8][i & 255] = 0;
  __syncthreads();
  for (int t = wid; t < T; t += NW) {
    if (tagged)
      topk_warp_tagged(tagged, TS, gen, has_gate, t, E, k, S.idx, S.w, S.sg, user_idx, user_w,
                       rb, wctl, status);
    else
      topk_warp<false>(logits, gate_logit, t, E, k, S.idx, S.w, S.sg, user_idx, user_w, rb);
  }
  __syncthreads();
  const int N = T * k;
  const int e_a = tid < N ? S.idx[tid] : -1;
  if (e_a >= 0) atomicAdd(&S.cnt[e_a], 1);
  __syncthreads();
  // exclusive scans of the counts and of the sub-slot counts over experts
  const int c = tid < E ? S.cnt[tid] : 0;
  const int ns = (c + 7) >> 3;
  int ic = c, isub = ns;
  if (tid < 256) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y1 = __shfl_up_sync(0xffffffffu, ic, o);
      const int y2 = __shfl_up_sync(0xffffffffu, isub, o);
      if (lane >= o) {
        ic += y1;
        isub += y2;
      }
    }
    if (lane == 31) {
      S.wsum[wid] = ic;
      S.wsub[wid] = isub;
    }
  }
  __syncthreads();
  if (tid < 256) {
    int pc = 0, ps = 0;
    for (int i = 0; i < wid; ++i) {
      pc += S.wsum[i];
      ps += S.wsub[i];
    }
    S.off[tid] = pc + ic - c;
    S.sbase[tid] = ps + isub - ns;
    if (tid == 0) {
      int tot = 0;
      for (int i = 0; i < 8; ++i) tot += S.wsub[i];
      S.nss = tot;
    }
  }
  // stable scatter: rank among the same expert's assignments, in id order
  unsigned peers = 0;
  if (tid < 256) {
    peers = __match_any_sync(0xffffffffu, e_a);
    if (e_a >= 0 && (__ffs(peers) - 1) == lane) wc[wid][e_a] = __popc(peers);
  }
  __syncthreads();
  if (tid < 256 && e_a >= 0) {
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int pre = 0;
    for (int i = 0; i < wid; ++i) pre += wc[i][e_a];
    S.perm[S.off[e_a] + pre + rank] = tid;
  }
  if (tid < E) {
    for (int i = 0; i < ns; ++i) {
      const int ss = S.sbase[tid] + i;
      S.ss_e[ss] = tid;
      S.ss_off[ss] = S.off[tid] + 8 * i;
      S.ss_cnt[ss] = min(8, c - 8 * i);
    }
  }
  __syncthreads();
}

}  // namespace moe
