// route.cu -- standalone routing kernels (router logits, top-k + weights,
// bucketing, slots) over the device functions of route.cuh.

#include "route.cuh"

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

__global__ void __launch_bounds__(256) k_subslots(const int32_t* __restrict__ offsets, int E,
                                                  int* nss, int* se, int* so, int* sc,
                                                  int run, int cmin, int cmax) {
  __shared__ int wcount[8];
  subslots_cta(offsets, E, nss, se, so, sc, wcount, run, cmin, cmax);
}

// ---------------------------------------------------------------------------
// Router logits of a prefill window on the tensor cores: a dense contraction
// logits[T, E + 1] = x[T, H] * W[E + 1, H]^T (row E the shared-gate row).
// Every weight w (fp32, or an affine-8 value fma(s, q, b) in fp32) is split
// exactly into three bf16 parts w = w1 + w2 + w3 (8 significant bits each, the
// remainders exact in fp32); bf16 activations are exact operands, fp16 ones
// split exactly into two bf16 parts.  So every product is exact and the sums
// are fp32 (mma.sync m16n8k16, fp32 accumulation).  A block computes a tile of
// 32 tokens x 32 rows over 64-column chunks of H staged in shared memory; warp
// w takes tokens 16 (w & 1) .. and rows 16 (w >> 1) .. (two 8-row n-tiles).
constexpr int kRtTok = 32, kRtRows = 32, kRtK = 64, kRtPitch = kRtK + 8;  // bf16 elements
constexpr int kRtSplit = 4;  // k-slices per tile, summed in order by k_router_sum

__device__ __forceinline__ void split3_bf16(float v, uint16_t& a, uint16_t& b, uint16_t& c) {
  const __nv_bfloat16 h1 = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(h1);
  const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(h2);
  a = __bfloat16_as_ushort(h1);
  b = __bfloat16_as_ushort(h2);
  c = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
}

// blockIdx.z: k-slice of H; the slice's sums go to part[z][T][E + 1]
__global__ void __launch_bounds__(128) k_router_tc(const RouterJob J, float* part) {
  __shared__ __align__(16) uint16_t xs[2][kRtTok][kRtPitch];
  __shared__ __align__(16) uint16_t wsm[3][kRtRows][kRtPitch];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int t0 = blockIdx.x * kRtTok, r0 = blockIdx.y * kRtRows;
  const int nrows = J.E + (J.gq ? 1 : 0);
  const int px = J.f16 ? 2 : 1;  // bf16 parts of x
  const bool w1part = J.round_bf16 || (!J.gq && J.fmt == MOE_FMT_BF16);
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  const int kslice = J.H / kRtSplit;
  for (int k0 = blockIdx.z * kslice; k0 < (blockIdx.z + 1) * kslice; k0 += kRtK) {
    // x chunk: 32 tokens x 64 columns, 16 values per thread
    {
      const int tk = tid >> 2, c = (tid & 3) * 16;
      const int tok = t0 + tk;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (tok < J.T) v = *reinterpret_cast<const uint4*>(J.x + size_t(tok) * J.H + k0 + c + 8 * h);
        if (!J.f16) {
          *reinterpret_cast<uint4*>(&xs[0][tk][c + 8 * h]) = v;
        } else {  // fp16 -> exact bf16 hi + lo
          const uint32_t in[4] = {v.x, v.y, v.z, v.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&in[j]));
            const __nv_bfloat162 bh = __floats2bfloat162_rn(f.x, f.y);
            const float2 fh = __bfloat1622float2(bh);
            const __nv_bfloat162 bl = __floats2bfloat162_rn(f.x - fh.x, f.y - fh.y);
            hi[j] = *reinterpret_cast<const uint32_t*>(&bh);
            lo[j] = *reinterpret_cast<const uint32_t*>(&bl);
          }
          *reinterpret_cast<uint4*>(&xs[0][tk][c + 8 * h]) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(&xs[1][tk][c + 8 * h]) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    }
    // weight chunk: 32 rows x 64 columns, 16 values per thread, split in 3
    {
      const int rr = tid >> 2, c = (tid & 3) * 16;
      const int row = r0 + rr;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float w[4] = {0.f, 0.f, 0.f, 0.f};
        const int k = k0 + c + 4 * q4;
        if (row < nrows) {
          if (row >= J.E)
            router_load_w4(J.gfmt, J.gq, J.gs, J.gb, 0, J.H, k, w, J.round_bf16 != 0);
          else
            router_load_w4(J.fmt, J.q, J.s, J.b, row, J.H, k, w, J.round_bf16 != 0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          split3_bf16(w[j], wsm[0][rr][c + 4 * q4 + j], wsm[1][rr][c + 4 * q4 + j],
                      wsm[2][rr][c + 4 * q4 + j]);
      }
    }
    __syncthreads();
    const int tb = 16 * (warp & 1), rb = 16 * (warp >> 1);
#pragma unroll
    for (int kk = 0; kk < kRtK; kk += 16) {
#pragma unroll
      for (int xp = 0; xp < 2; ++xp) {
        if (xp >= px) break;
        const uint32_t a0 = *reinterpret_cast<const uint32_t*>(&xs[xp][tb + g][kk + 2 * t4]);
        const uint32_t a1 = *reinterpret_cast<const uint32_t*>(&xs[xp][tb + g + 8][kk + 2 * t4]);
        const uint32_t a2 = *reinterpret_cast<const uint32_t*>(&xs[xp][tb + g][kk + 2 * t4 + 8]);
        const uint32_t a3 =
            *reinterpret_cast<const uint32_t*>(&xs[xp][tb + g + 8][kk + 2 * t4 + 8]);
#pragma unroll
        for (int wp = 0; wp < 3; ++wp) {
          if (wp > 0 && w1part) break;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int rw = rb + 8 * nt + g;
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&wsm[wp][rw][kk + 2 * t4]);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&wsm[wp][rw][kk + 2 * t4 + 8]);
            mma16816<false>(acc[nt], a0, a1, a2, a3, b0, b1);
          }
        }
      }
    }
    __syncthreads();
  }
  // acc[nt]: (token tb + g, rows rb + 8 nt + 2 t4, +1), (token tb + g + 8, same rows)
  const int tb = 16 * (warp & 1), rb = 16 * (warp >> 1);
  float* pz = part + size_t(blockIdx.z) * J.T * nrows;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = t0 + tb + g + 8 * (i >> 1);
      const int row = r0 + rb + 8 * nt + 2 * t4 + (i & 1);
      if (tok < J.T && row < nrows) pz[size_t(tok) * nrows + row] = acc[nt][i];
    }
}

// logits = the k-slices' sums added in slice order, plus the bias
__global__ void k_router_sum(const RouterJob J, const float* __restrict__ part) {
  const int nrows = J.E + (J.gq ? 1 : 0);
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= long(J.T) * nrows) return;
  const int tok = int(i / nrows), row = int(i - long(tok) * nrows);
  const size_t stride = size_t(J.T) * nrows;
  float v = part[i];
#pragma unroll
  for (int z = 1; z < kRtSplit; ++z) v += part[i + z * stride];
  if (row < J.E)
    J.logits[size_t(tok) * J.E + row] = v + (J.bias ? J.bias[row] : 0.f);
  else
    J.gate_logit[tok] = v;
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
  if (J.T > kRouterTensorMin && J.part && J.H % (kRtK * kRtSplit) == 0) {
    k_router_tc<<<dim3((J.T + kRtTok - 1) / kRtTok, (rows + kRtRows - 1) / kRtRows, kRtSplit), 128,
                  0, st>>>(J, J.part);
    const long n = long(J.T) * rows;
    k_router_sum<<<unsigned((n + 255) / 256), 256, 0, st>>>(J, J.part);
  } else
    k_router<1><<<dim3(rows, (J.T + kRouterTT - 1) / kRouterTT), 32 * KS, 0, st>>>(J, KS);
  return cudaGetLastError();
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

}  // namespace moe
