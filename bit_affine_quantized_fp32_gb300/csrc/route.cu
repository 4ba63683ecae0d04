// route.cu -- standalone routing kernels (router logits, top-k + weights,
// bucketing, slots) over the device functions of route.cuh.

#include "route.cuh"
#include "host.h"

namespace moe {

namespace {

// Above this many tokens the logits are a tensor-core contraction
// (k_router_tc); up to it (the decode form) the CUDA-core router gives the
// bits the fused decode kernel gives.
constexpr int kRouterTensorMin = 32;

// blockIdx.x: block of R router rows, blockIdx.y: run of kRouterTT tokens;
// KS warps (one k-split each)
template <int R>
__global__ void __launch_bounds__(256) k_router(const RouterJob J, int KS) {
  __shared__ float part[R * 8 * kRouterTT];
  const int t0 = blockIdx.y * kRouterTT;
  router_block_rows<R>(J, KS, blockIdx.x, part, t0, min(kRouterTT, J.T - t0));
}

__global__ void k_topk(const float* __restrict__ logits, const float* __restrict__ gate_logit,
                       int T, int E, int k, int32_t* __restrict__ idx, float* __restrict__ w,
                       float* __restrict__ sg, int rb) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_warp<false>(logits, gate_logit, t, E, k, idx, w, sg, nullptr, nullptr, rb != 0);
}

__global__ void __launch_bounds__(1024) k_bucket(const int32_t* __restrict__ idx, int N, int E,
                                                 int32_t* __restrict__ offsets,
                                                 int32_t* __restrict__ perm) {
  __shared__ BucketSmem S;
  bucket_cta(idx, N, E, offsets, perm, S);
}

// k_bucket followed, in the same block, by the two tables of k_subslots_pair
// (the offsets it reads are the block's own writes, visible after the
// barrier).
__global__ void __launch_bounds__(1024) k_bucket_tables(const int32_t* __restrict__ idx, int N,
                                                        int E, int32_t* __restrict__ offsets,
                                                        int32_t* __restrict__ perm, int split,
                                                        SubslotTable A, int run_a, SubslotTable B,
                                                        int run_b) {
  __shared__ BucketSmem S;
  __shared__ int wcount[8];
  bucket_cta(idx, N, E, offsets, perm, S);
  __syncthreads();
  subslots_cta(offsets, E, A.n, A.e, A.off, A.cnt, wcount, run_a, split, 1 << 30);
  subslots_cta(offsets, E, B.n, B.e, B.off, B.cnt, wcount, run_b, 0, split);
}

__global__ void __launch_bounds__(256) k_subslots(const int32_t* __restrict__ offsets, int E,
                                                  int* nss, int* se, int* so, int* sc,
                                                  int run, int cmin, int cmax) {
  __shared__ int wcount[8];
  subslots_cta(offsets, E, nss, se, so, sc, wcount, run, cmin, cmax);
}

// Both tables of a prefill call in one launch: runs of `run_a` positions of
// the experts with more than `split` assignments, runs of `run_b` of the
// others (as two k_subslots launches).
__global__ void __launch_bounds__(256) k_subslots_pair(const int32_t* __restrict__ offsets, int E,
                                                       int split, SubslotTable A, int run_a,
                                                       SubslotTable B, int run_b) {
  __shared__ int wcount[8];
  subslots_cta(offsets, E, A.n, A.e, A.off, A.cnt, wcount, run_a, split, 1 << 30);
  subslots_cta(offsets, E, B.n, B.e, B.off, B.cnt, wcount, run_b, 0, split);
}

// ---------------------------------------------------------------------------
// Router logits of a prefill window on the tensor cores: a dense contraction
// logits[T, E + 1] = x[T, H] * W[E + 1, H]^T (row E the shared-gate row).
// Every weight w (fp32, or an affine-8 value fma(s, q, b) in fp32) is split
// exactly into three bf16 parts w = w1 + w2 + w3 (8 significant bits each, the
// remainders exact in fp32); bf16 activations are exact operands, fp16 ones
// split exactly into two bf16 parts.  So every product is exact and the sums
// are fp32 (mma.sync m16n8k16, fp32 accumulation).  k_router_split writes the
// parts once per call (workspace); a k_router_tc block computes a tile of 64
// tokens x 32 rows over a k-slice of H, streaming 64-column chunks of the
// parts through a ring of kRtStages shared-memory stages (cp.async); warp w
// takes tokens 32 (w & 1) .. (two 16-row m-tiles) and rows 16 (w >> 1) ..
// (two 8-row n-tiles): four accumulator chains, each fragment loaded once
// for two or three MMAs.
constexpr int kRtTok = 64, kRtRows = 32, kRtK = 64, kRtPitch = kRtK + 8;  // bf16 elements
constexpr int kRtSplit = 4;   // k-slices per tile, summed in order by k_topk_parts
constexpr int kRtStages = 4;  // chunks in flight per block
constexpr int kRtXPart = kRtTok * kRtPitch;   // elements of one x-part tile
constexpr int kRtWPart = kRtRows * kRtPitch;  // elements of one weight-part tile

__device__ __forceinline__ void split3_bf16(float v, uint16_t& a, uint16_t& b, uint16_t& c) {
  const __nv_bfloat16 h1 = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(h1);
  const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(h2);
  a = __bfloat16_as_ushort(h1);
  b = __bfloat16_as_ushort(h2);
  c = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
}

// rows whose weights are one exact bf16 part (the chain's bf16 rows, or bf16
// router rows without a gate row of another format)
__host__ __device__ inline bool router_one_part(const RouterJob& J) {
  return J.round_bf16 || (!J.gq && J.fmt == MOE_FMT_BF16);
}

// wp[p][r][k] (p < 3, r < E + gate) = part p of weight (r, k); for fp16
// activations xp[p][t][k] (p < 2) = part p of x (t, k).  Thread: 4 columns.
__global__ void k_router_split(const RouterJob J, uint16_t* __restrict__ wp,
                               uint16_t* __restrict__ xp) {
  const int nrows = J.E + (J.gq ? 1 : 0);
  const int q4 = J.H / 4;
  const long nw = long(nrows) * q4;
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < nw) {
    const int r = int(i / q4), k = int(i - long(r) * q4) * 4;
    float w[4];
    if (r >= J.E)
      router_load_w4(J.gfmt, J.gq, J.gs, J.gb, 0, J.H, k, w, J.round_bf16 != 0);
    else
      router_load_w4(J.fmt, J.q, J.s, J.b, r, J.H, k, w, J.round_bf16 != 0);
    uint16_t a[4], b[4], c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) split3_bf16(w[j], a[j], b[j], c[j]);
    const size_t o = size_t(r) * J.H + k, ps = size_t(nrows) * J.H;
    auto put = [&](uint16_t* dst, const uint16_t (&v)[4]) {
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(uint32_t(v[0]) | (uint32_t(v[1]) << 16), uint32_t(v[2]) | (uint32_t(v[3]) << 16));
    };
    put(wp + o, a);
    put(wp + ps + o, b);
    put(wp + 2 * ps + o, c);
    return;
  }
  if (!J.f16) return;
  const long j = i - nw;
  if (j >= long(J.T) * q4) return;
  const int t = int(j / q4), k = int(j - long(t) * q4) * 4;
  const uint2 v = *reinterpret_cast<const uint2*>(J.x + size_t(t) * J.H + k);
  const uint32_t in[2] = {v.x, v.y};
  uint32_t hi[2], lo[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&in[h]));
    const __nv_bfloat162 bh = __floats2bfloat162_rn(f.x, f.y);
    const float2 fh = __bfloat1622float2(bh);
    const __nv_bfloat162 bl = __floats2bfloat162_rn(f.x - fh.x, f.y - fh.y);
    hi[h] = *reinterpret_cast<const uint32_t*>(&bh);
    lo[h] = *reinterpret_cast<const uint32_t*>(&bl);
  }
  const size_t o = size_t(t) * J.H + k;
  *reinterpret_cast<uint2*>(xp + o) = make_uint2(hi[0], hi[1]);
  *reinterpret_cast<uint2*>(xp + size_t(J.T) * J.H + o) = make_uint2(lo[0], lo[1]);
}

// Shared memory of one k_router_tc stage: px x-part tiles then nwp weight-part
// tiles.
__host__ __device__ inline int router_stage_elems(const RouterJob& J) {
  return (J.f16 ? 2 : 1) * kRtXPart + (router_one_part(J) ? 1 : 3) * kRtWPart;
}

// blockIdx.z: k-slice of H; the slice's sums go to part[z][T][E + 1]
__global__ void __launch_bounds__(128) k_router_tc(const RouterJob J, const uint16_t* __restrict__ wp,
                                                   const uint16_t* __restrict__ xp,
                                                   float* __restrict__ part) {
  extern __shared__ __align__(16) uint16_t rt_smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int t0 = blockIdx.x * kRtTok, r0 = blockIdx.y * kRtRows;
  const int nrows = J.E + (J.gq ? 1 : 0);
  const int px = J.f16 ? 2 : 1;                 // bf16 parts of x
  const int nwp = router_one_part(J) ? 1 : 3;   // bf16 parts of the weights
  const int SE = px * kRtXPart + nwp * kRtWPart;  // elements per stage
  const size_t ps = size_t(nrows) * J.H;
  const int kslice = J.H / kRtSplit, nchunk = kslice / kRtK, kbeg = blockIdx.z * kslice;
  // chunk c -> stage c % kRtStages: 16-byte pieces (row piece >> 3, columns
  // 8 (piece & 7) ..), thread tid taking pieces tid + 128 i; rows past T or
  // E + gate are left as they are (their products only reach sums that are
  // not written)
  auto issue = [&](int c) {
    uint16_t* S = rt_smem + (c % kRtStages) * SE;
    const int k0 = kbeg + c * kRtK;
#pragma unroll
    for (int h = 0; h < kRtTok * 8 / 128; ++h) {
      const int pc = tid + 128 * h, rr = pc >> 3, c8 = (pc & 7) * 8;
      for (int p = 0; p < px; ++p)
        if (t0 + rr < J.T) {
          const uint16_t* src = (J.f16 ? xp + size_t(p) * J.T * J.H : J.x) +
                                size_t(t0 + rr) * J.H + k0 + c8;
          cp_async16(S + p * kRtXPart + rr * kRtPitch + c8, src);
        }
    }
    uint16_t* W = S + px * kRtXPart;
#pragma unroll
    for (int h = 0; h < kRtRows * 8 / 128; ++h) {
      const int pc = tid + 128 * h, rr = pc >> 3, c8 = (pc & 7) * 8;
      for (int p = 0; p < nwp; ++p)
        if (r0 + rr < nrows)
          cp_async16(W + p * kRtWPart + rr * kRtPitch + c8,
                     wp + p * ps + size_t(r0 + rr) * J.H + k0 + c8);
    }
  };
  float acc[2][2][4] = {};
  for (int c = 0; c < kRtStages - 1; ++c) {
    if (c < nchunk) issue(c);
    cp_async_commit();
  }
  const int tb = 32 * (warp & 1), rb = 16 * (warp >> 1);
  for (int c = 0; c < nchunk; ++c) {
    if (c + kRtStages - 1 < nchunk) issue(c + kRtStages - 1);
    cp_async_commit();
    cp_async_wait<kRtStages - 1>();  // chunk c has landed (this thread's pieces)
    __syncthreads();
    const uint16_t* S = rt_smem + (c % kRtStages) * SE;
#pragma unroll
    for (int kk = 0; kk < kRtK; kk += 16) {
      uint32_t bw[3][2][2];  // [part][n-tile][reg]
#pragma unroll
      for (int wq = 0; wq < 3; ++wq) {
        if (wq >= nwp) break;
        const uint16_t* W = S + px * kRtXPart + wq * kRtWPart;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int rw = rb + 8 * nt + g;
          bw[wq][nt][0] = *reinterpret_cast<const uint32_t*>(W + rw * kRtPitch + kk + 2 * t4);
          bw[wq][nt][1] = *reinterpret_cast<const uint32_t*>(W + rw * kRtPitch + kk + 2 * t4 + 8);
        }
      }
#pragma unroll
      for (int xq = 0; xq < 2; ++xq) {
        if (xq >= px) break;
        const uint16_t* X = S + xq * kRtXPart;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int tr = tb + 16 * mt + g;
          const uint32_t a0 = *reinterpret_cast<const uint32_t*>(X + tr * kRtPitch + kk + 2 * t4);
          const uint32_t a1 =
              *reinterpret_cast<const uint32_t*>(X + (tr + 8) * kRtPitch + kk + 2 * t4);
          const uint32_t a2 =
              *reinterpret_cast<const uint32_t*>(X + tr * kRtPitch + kk + 2 * t4 + 8);
          const uint32_t a3 =
              *reinterpret_cast<const uint32_t*>(X + (tr + 8) * kRtPitch + kk + 2 * t4 + 8);
#pragma unroll
          for (int wq = 0; wq < 3; ++wq) {
            if (wq >= nwp) break;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
              mma16816<false>(acc[mt][nt], a0, a1, a2, a3, bw[wq][nt][0], bw[wq][nt][1]);
          }
        }
      }
    }
    __syncthreads();  // the stage is refilled by a later issue
  }
  // acc[mt][nt]: (token tb + 16 mt + g, rows rb + 8 nt + 2 t4, +1), (token + 8, same rows)
  float* pz = part + size_t(blockIdx.z) * J.T * nrows;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int tok = t0 + tb + 16 * mt + g + 8 * (i >> 1);
        const int row = r0 + rb + 8 * nt + 2 * t4 + (i & 1);
        if (tok < J.T && row < nrows) pz[size_t(tok) * nrows + row] = acc[mt][nt][i];
      }
}

// Top-k of token t (one warp) from the k-slice sums: each logit is the
// slices' sums added in slice order, plus the bias; it is written to
// J.logits (and the gate logit to J.gate_logit) on the way.
__global__ void k_topk_parts(const RouterJob J, const float* __restrict__ part, int k,
                             int32_t* __restrict__ idx, float* __restrict__ w,
                             float* __restrict__ sg, int rb) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= J.T) return;
  const int lane = threadIdx.x & 31;
  const int nrows = J.E + (J.gq ? 1 : 0);
  const size_t stride = size_t(J.T) * nrows;
  const float* row = part + size_t(t) * nrows;
  unsigned long long key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * lane + i;
    key[i] = 0ull;
    if (e < J.E) {
      float v = __ldcg(row + e);
#pragma unroll
      for (int z = 1; z < kRtSplit; ++z) v += __ldcg(row + z * stride + e);
      v = v + (J.bias ? J.bias[e] : 0.f);
      J.logits[size_t(t) * J.E + e] = v;
      key[i] = rank_key(v, e);
    }
  }
  float gl = 0.f;
  if (J.gq) {
    gl = __ldcg(row + J.E);
#pragma unroll
    for (int z = 1; z < kRtSplit; ++z) gl += __ldcg(row + z * stride + J.E);
    if (lane == 0) J.gate_logit[t] = gl;
  }
  topk_select(key, t, k, idx, w, sg, J.gq != nullptr, gl, nullptr, nullptr, rb != 0);
}

}  // namespace

// k-splits of a router row: the fewest with at most 2 x 128 columns per warp
// (short dependent chains), else at most 4 x 128.
int router_ks(int H) {
  for (int ks = 1; ks <= 8; ks <<= 1)
    if (H % (ks * 128) == 0 && H / (ks * 128) <= 2) return ks;
  for (int ks = 1; ks <= 8; ks <<= 1)
    if (H % (ks * 128) == 0 && H / (ks * 128) <= 4) return ks;
  return 0;
}

int router_blocks(int E, bool gate, int H) {
  const int KS = router_ks(H);
  if (KS == 0) return 0;
  const int RPB = 8 / KS;
  return (E + (gate ? 1 : 0) + RPB - 1) / RPB;
}

cudaError_t launch_router(const RouterJob& J, cudaStream_t st) {
  if (J.T <= 0) return cudaSuccess;
  const int KS = router_ks(J.H);
  if (KS == 0) return cudaErrorInvalidValue;
  const int rows = J.E + (J.gq ? 1 : 0);
  k_router<1><<<dim3(rows, (J.T + kRouterTT - 1) / kRouterTT), 32 * KS, 0, st>>>(J, KS);
  return cudaGetLastError();
}

// Router and top-k: above kRouterTensorMin tokens (with the scratch) the
// tensor-core router's k-slice sums go straight into the top-k, else the SIMT
// router's logits through k_topk.
cudaError_t launch_router_topk(const RouterJob& J, int k, int32_t* idx, float* w, float* sg,
                               bool round_bf16, cudaStream_t st) {
  if (J.T <= 0) return cudaSuccess;
  const int rows = J.E + (J.gq ? 1 : 0);
  if (J.T > kRouterTensorMin && J.part && J.split && J.H % (kRtK * kRtSplit) == 0 &&
      router_ks(J.H) != 0) {
    const long n_split = long(rows) * (J.H / 4) + (J.f16 ? long(J.T) * (J.H / 4) : 0);
    k_router_split<<<unsigned((n_split + 255) / 256), 256, 0, st>>>(J, J.split,
                                                                    J.split + 3 * size_t(rows) * J.H);
    const int smem = kRtStages * router_stage_elems(J) * 2;
    const cudaError_t e = ensure_dynamic_smem((const void*)k_router_tc, smem);
    if (e != cudaSuccess) return e;
    k_router_tc<<<dim3((J.T + kRtTok - 1) / kRtTok, (rows + kRtRows - 1) / kRtRows, kRtSplit), 128,
                  smem, st>>>(J, J.split, J.split + 3 * size_t(rows) * J.H, J.part);
    k_topk_parts<<<(J.T + 7) / 8, 256, 0, st>>>(J, J.part, k, idx, w, J.gq ? sg : nullptr,
                                                round_bf16 ? 1 : 0);
    return cudaGetLastError();
  }
  cudaError_t e = launch_router(J, st);
  if (e != cudaSuccess) return e;
  return launch_topk(J.logits, J.gq ? J.gate_logit : nullptr, J.T, J.E, k, idx, w,
                     J.gq ? sg : nullptr, round_bf16, st);
}

cudaError_t launch_topk(const float* logits, const float* gate_logit, int T, int E, int k,
                        int32_t* idx, float* w, float* sg, bool round_bf16, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  k_topk<<<(T + 7) / 8, 256, 0, st>>>(logits, gate_logit, T, E, k, idx, w, sg, round_bf16);
  return cudaGetLastError();
}

cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* offsets,
                          int32_t* perm, cudaStream_t st) {
  k_bucket<<<1, 1024, 0, st>>>(idx, T * k, E, offsets, perm);
  return cudaGetLastError();
}

cudaError_t launch_subslots(const int32_t* offsets, int E, int* nss, int* se, int* so, int* sc,
                            cudaStream_t st, int run, int cmin, int cmax) {
  k_subslots<<<1, 256, 0, st>>>(offsets, E, nss, se, so, sc, run, cmin, cmax);
  return cudaGetLastError();
}

cudaError_t launch_bucket_tables(const int32_t* idx, int T, int k, int E, int32_t* offsets,
                                 int32_t* perm, int split, const SubslotTable& A, int run_a,
                                 const SubslotTable& B, int run_b, cudaStream_t st) {
  k_bucket_tables<<<1, 1024, 0, st>>>(idx, T * k, E, offsets, perm, split, A, run_a, B, run_b);
  return cudaGetLastError();
}

cudaError_t launch_subslots_pair(const int32_t* offsets, int E, int split, const SubslotTable& A,
                                 int run_a, const SubslotTable& B, int run_b, cudaStream_t st) {
  k_subslots_pair<<<1, 256, 0, st>>>(offsets, E, split, A, run_a, B, run_b);
  return cudaGetLastError();
}

}  // namespace moe
