// route.cu -- router logits, top-k with routing weights, and token->expert
// bucketing.
//
// Source: "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803",
// comment "Progress on the 4-bit gate": fp32 logits over the experts and the
// shared expert's gate row, top-k by logit with ties to the lower id, weights
// exp(l - l_top) over the k (normalised over the k here), the shared expert
// weighted by sigmoid(gate).  Bucketing (a stable counting sort of the
// assignments by expert) serves the grouped experts of "Sage-A1.5 ... on the
// XPU backend #1329" (Proposal: grouped MoE).

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRouterTT = 64;  // tokens per CTA row-tile

// Four consecutive weights of row r at column k (k % 4 == 0) as fp32.
__device__ __forceinline__ void load_w4(int fmt, const void* q, const uint16_t* s,
                                        const uint16_t* b, int r, int H, int k, float (&w)[4]) {
  if (fmt == MOE_FMT_F32) {
    const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(q) + size_t(r) * H + k);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if (fmt == MOE_FMT_BF16 || fmt == MOE_FMT_F16) {
    const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(q) + size_t(r) * H + k);
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
}

// Each warp owns (row, k-split q) and keeps its 4*NI weights in registers;
// the KS partial sums of a row are added in a fixed order.
template <int NI>
__global__ void __launch_bounds__(256) k_router(const RouterJob J, int KS) {
  __shared__ float part[8][kRouterTT];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int RPB = 8 / KS;
  const int rl = wid / KS, q = wid - rl * KS;
  const int row = blockIdx.x * RPB + rl;
  const int nrows = J.E + (J.gq ? 1 : 0);
  const int t0 = blockIdx.y * kRouterTT;
  const int tn = min(kRouterTT, J.T - t0);
  const bool active = row < nrows;
  const int kq = q * (J.H / KS);
  float w[NI][4];
  if (active) {
    const bool gate = row >= J.E;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int k = kq + 128 * i + 4 * lane;
      if (gate)
        load_w4(J.gfmt, J.gq, J.gs, J.gb, 0, J.H, k, w[i]);
      else
        load_w4(J.fmt, J.q, J.s, J.b, row, J.H, k, w[i]);
    }
  }
  for (int tl = 0; tl < tn; ++tl) {
    float acc = 0.f;
    if (active) {
      const uint16_t* xr = J.x + size_t(t0 + tl) * J.H;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const uint2 v = *reinterpret_cast<const uint2*>(xr + kq + 128 * i + 4 * lane);
        acc = fmaf(w[i][0], act_to_float(uint16_t(v.x & 0xFFFF), J.f16), acc);
        acc = fmaf(w[i][1], act_to_float(uint16_t(v.x >> 16), J.f16), acc);
        acc = fmaf(w[i][2], act_to_float(uint16_t(v.y & 0xFFFF), J.f16), acc);
        acc = fmaf(w[i][3], act_to_float(uint16_t(v.y >> 16), J.f16), acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) part[wid][tl] = acc;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < RPB * tn; i += blockDim.x) {
    const int r2 = i / tn, tl = i - r2 * tn;
    const int row2 = blockIdx.x * RPB + r2;
    if (row2 >= nrows) continue;
    float s = 0.f;
    for (int qq = 0; qq < KS; ++qq) s += part[r2 * KS + qq][tl];
    if (row2 < J.E) {
      if (J.bias) s += J.bias[row2];
      J.logits[size_t(t0 + tl) * J.E + row2] = s;
    } else {
      J.gate_logit[t0 + tl] = s;
    }
  }
}

// One warp per token: k rounds of a warp-wide arg-best over the remaining
// experts (each lane holds experts lane, lane+32, ...), then the weights.
__global__ void k_topk(const float* __restrict__ logits, const float* __restrict__ gate_logit,
                       int T, int E, int k, int32_t* __restrict__ idx, float* __restrict__ w,
                       float* __restrict__ sg) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float v[8];
  bool ok[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    ok[i] = e < E;
    v[i] = ok[i] ? logits[size_t(t) * E + e] : 0.f;
  }
  int sel_e[8];
  float sel_v[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    sel_e[r] = 0;
    sel_v[r] = 0.f;
    if (r < k) {
      int be = -1;
      float bv = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        if (ok[i] && (be < 0 || ranks_before(v[i], e, bv, be))) {
          be = e;
          bv = v[i];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        if (oe >= 0 && (be < 0 || ranks_before(ov, oe, bv, be))) {
          be = oe;
          bv = ov;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (lane + 32 * i == be) ok[i] = false;
      sel_e[r] = be;
      sel_v[r] = bv;
    }
  }
  if (lane == 0) {
    const float top = sel_v[0];
    float ex[8];
    float den = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      ex[r] = r < k ? expf(sel_v[r] - top) : 0.f;
      if (r < k) den += ex[r];
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (r < k) {
        idx[size_t(t) * k + r] = sel_e[r];
        w[size_t(t) * k + r] = ex[r] / den;
      }
    }
    if (gate_logit && sg) sg[t] = 1.f / (1.f + expf(-gate_logit[t]));
  }
}

// Stable counting sort of the N = T*k assignment ids by expert (one CTA).
// Inside a 1024-assignment chunk, the rank of an assignment among the same
// expert's is found with warp match + per-warp counts; chunks go in order.
__global__ void __launch_bounds__(1024) k_bucket(const int32_t* __restrict__ idx, int N, int E,
                                                 int32_t* __restrict__ offsets,
                                                 int32_t* __restrict__ perm) {
  __shared__ int cnt[256];
  __shared__ int cur[256];
  __shared__ int wsum[8];
  __shared__ int wc[32][256];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid < 256) cnt[tid] = 0;
  __syncthreads();
  for (int a = tid; a < N; a += 1024) {
    const int e = idx[a];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  int incl = 0;
  if (tid < 256) {
    incl = tid < E ? cnt[tid] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[wid] = incl;
  }
  __syncthreads();
  if (tid < 256) {
    int pre = 0;
    for (int i = 0; i < wid; ++i) pre += wsum[i];
    incl += pre;
    const int c = tid < E ? cnt[tid] : 0;
    cur[tid] = incl - c;
    if (tid < E) offsets[tid + 1] = incl;
    if (tid == 0) offsets[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < N; base += 1024) {
    for (int i = lane; i < 256; i += 32) wc[wid][i] = 0;
    __syncwarp();
    const int a = base + tid;
    int e = a < N ? idx[a] : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const bool leader = (__ffs(peers) - 1) == lane;
    if (e >= 0 && leader) wc[wid][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int pre = 0;
      for (int i = 0; i < wid; ++i) pre += wc[i][e];
      perm[cur[e] + pre + rank] = a;
    }
    __syncthreads();
    if (tid < E) {
      int tot = 0;
      for (int i = 0; i < 32; ++i) tot += wc[i][tid];
      cur[tid] += tot;
    }
    __syncthreads();
  }
}

// Active-expert slots (ascending id) from the bucket offsets, and the token of
// every bucket position.
__global__ void __launch_bounds__(256) k_slots(const int32_t* __restrict__ offsets,
                                               const int32_t* __restrict__ perm, int P, int k,
                                               int E, int* __restrict__ nslots,
                                               int* __restrict__ se, int* __restrict__ so,
                                               int* __restrict__ sc, int* __restrict__ blist) {
  __shared__ int wcount[8];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int c = tid < E ? offsets[tid + 1] - offsets[tid] : 0;
  const bool f = c > 0;
  const unsigned m = __ballot_sync(0xffffffffu, f);
  if (lane == 0) wcount[wid] = __popc(m);
  __syncthreads();
  int pre = 0;
  for (int i = 0; i < wid; ++i) pre += wcount[i];
  if (f) {
    const int s = pre + __popc(m & ((1u << lane) - 1u));
    se[s] = tid;
    so[s] = offsets[tid];
    sc[s] = c;
  }
  if (tid == 0) {
    int tot = 0;
    for (int i = 0; i < 8; ++i) tot += wcount[i];
    *nslots = tot;
  }
  for (int p = tid; p < P; p += 256) blist[p] = perm[p] / k;
}

}  // namespace

int router_ks(int H) {
  for (int ks = 1; ks <= 8; ks <<= 1)
    if (H % (ks * 128) == 0 && H / (ks * 128) <= 4) return ks;
  return 0;
}

cudaError_t launch_router(const RouterJob& J, cudaStream_t st) {
  if (J.T <= 0) return cudaSuccess;
  const int KS = router_ks(J.H);
  if (KS == 0) return cudaErrorInvalidValue;
  const int NI = J.H / (KS * 128);
  const int RPB = 8 / KS;
  const int nrows = J.E + (J.gq ? 1 : 0);
  dim3 grid((nrows + RPB - 1) / RPB, (J.T + kRouterTT - 1) / kRouterTT);
  switch (NI) {
    case 1: k_router<1><<<grid, 256, 0, st>>>(J, KS); break;
    case 2: k_router<2><<<grid, 256, 0, st>>>(J, KS); break;
    case 3: k_router<3><<<grid, 256, 0, st>>>(J, KS); break;
    default: k_router<4><<<grid, 256, 0, st>>>(J, KS); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, const float* gate_logit, int T, int E, int k,
                        int32_t* idx, float* w, float* sg, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  k_topk<<<(T + 7) / 8, 256, 0, st>>>(logits, gate_logit, T, E, k, idx, w, sg);
  return cudaGetLastError();
}

cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* offsets,
                          int32_t* perm, cudaStream_t st) {
  k_bucket<<<1, 1024, 0, st>>>(idx, T * k, E, offsets, perm);
  return cudaGetLastError();
}

cudaError_t launch_slots(const int32_t* offsets, const int32_t* perm, int T, int k, int E,
                         int* nslots, int* slot_e, int* slot_off, int* slot_cnt, int* blist,
                         cudaStream_t st) {
  k_slots<<<1, 256, 0, st>>>(offsets, perm, T * k, k, E, nslots, slot_e, slot_off, slot_cnt,
                             blist);
  return cudaGetLastError();
}

}  // namespace moe
