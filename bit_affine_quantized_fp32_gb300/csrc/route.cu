// route.cu -- standalone routing kernels (router logits, top-k + weights,
// bucketing, slots) over the device functions of route.cuh.

#include "route.cuh"

namespace moe {

namespace {

// blockIdx.x: router block (rows), blockIdx.y: run of kRouterTT tokens
__global__ void __launch_bounds__(256) k_router(const RouterJob J, int KS) {
  __shared__ float part[8 * kRouterTT];
  const int t0 = blockIdx.y * kRouterTT;
  router_block(J, KS, blockIdx.x, part, J.x + size_t(t0) * J.H, t0, min(kRouterTT, J.T - t0));
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
  k_router<<<dim3(router_blocks(J.E, J.gq != nullptr, J.H), (J.T + kRouterTT - 1) / kRouterTT),
             256, 0, st>>>(J, KS);
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
