// units.cu -- standalone decode-path expert kernels: the item engine
// (engine.cuh) over one matrix family per launch (gate/up units with the
// SwiGLU epilogue, or down units), the per-64-group sums of the activations,
// and the weighted combine.  The fused layer kernel (decode.cu) runs the same
// device functions per unit, so both paths give the same bits.
//
// Source: "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803",
// comment "Progress on the 4-bit gate": grouped affine experts with a SwiGLU
// epilogue, decode rows summed in fp32, the slots' fma sum rounded once.

#include "kernels.h"

namespace moe {

namespace {

__device__ __forceinline__ int subslot_count(const SubSlots& S) {
  return S.n ? __ldcg(S.n) : (S.fixed_T + kMaxTok - 1) / kMaxTok;
}

// The units of this CTA: u = blockIdx.x + j * gridDim.x over n_subslots x
// blocks, sub-slot major.
struct JobSched {
  const UnitJob* J;
  int nblk, nu;
  __device__ explicit JobSched(const UnitJob* j) : J(j) {
    nblk = J->C.geo[J->mat].t.nblk;
    const int total = subslot_count(J->ss) * nblk;
    const int b = blockIdx.x, G = gridDim.x;
    nu = total > b ? (total - b + G - 1) / G : 0;
  }
  __device__ int n_units() const { return nu; }
  __device__ UnitInfo unit(int j) const {
    const int u = blockIdx.x + j * gridDim.x;
    const int ss = u / nblk;
    UnitInfo r;
    r.kind = (J->mat & 1) ? kItemDown : kItemGateUp;
    r.mat = J->mat;
    r.blk = u - ss * nblk;
    if (J->ss.n) {
      r.e = __ldcg(J->ss.e + ss);
      r.off = __ldcg(J->ss.off + ss);
      r.cnt = __ldcg(J->ss.cnt + ss);
    } else {
      r.e = J->ss.fixed_e;
      r.off = kMaxTok * ss;
      r.cnt = min(kMaxTok, J->ss.fixed_T - kMaxTok * ss);
    }
    r.nch = J->C.geo[J->mat].t.nch;
    r.rows = J->rows;
    r.signal = -1;
    r.wait_ctr = -1;
    r.wait_target = 0;
    return r;
  }
  __device__ const MatSource& source(int) const { return J->src; }
  __device__ const int* perm() const { return J->perm; }
  __device__ int topk() const { return J->k; }
  __device__ void combine(int) const {}
};

template <int FMT, bool F16A>
__global__ void __launch_bounds__(kEngineThreads, 1)
    k_units(const __grid_constant__ UnitJob J, int S, int SB) {
  extern __shared__ __align__(128) uint8_t stages[];
  __shared__ EngineSmem E;
  engine_init(E, S);
  fence_proxy_async();
  __syncthreads();
  const JobSched sch(&J);
  if ((threadIdx.x >> 5) == kProducerWarp)
    producer_run(J.C, E, stages, SB, S, sch, nullptr);
  else
    consumer_run<FMT, F16A>(J.C, E, stages, SB, S, sch, nullptr);
}

__global__ void k_xsum(const uint16_t* __restrict__ x, int T, int H, int f16, TileGeo g13,
                       float* __restrict__ xsum) {
  const int task = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (task >= T * (H >> 7)) return;
  xsum_task(x, H, f16 != 0, g13, xsum, task);
}

__global__ void __launch_bounds__(256) k_combine(const CombineArgs A) {
  combine_rows(A.y, A.w, A.ysh, A.sg, A.out, A.T, A.k, A.H, A.f16 != 0, blockIdx.x, threadIdx.x,
               blockDim.x);
}

template <int FMT, bool F16A>
cudaError_t launch_units_t(const UnitJob& J, int sms, cudaStream_t st) {
  const TileGeo geos[1] = {J.C.geo[J.mat].t};
  int S = 0, SB = 0;
  engine_stages(geos, 1, int(sizeof(EngineSmem)), &S, &SB);
  if (S < 2) return cudaErrorInvalidValue;
  const int smem = S * SB;
  // raise the dynamic shared-memory limit once per device (cudaFuncSetAttribute
  // is not a stream operation, so it stays out of captured graphs afterwards)
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] < smem) {
    e = cudaFuncSetAttribute(k_units<FMT, F16A>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  const int grid = J.max_units < sms ? J.max_units : sms;
  if (grid <= 0) return cudaSuccess;
  k_units<FMT, F16A><<<grid, kEngineThreads, smem, st>>>(J, S, SB);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_fmt(const UnitJob& J, bool f16a, int sms, cudaStream_t st) {
  return f16a ? launch_units_t<FMT, true>(J, sms, st) : launch_units_t<FMT, false>(J, sms, st);
}

}  // namespace

void engine_stages(const TileGeo* geos, int n, int static_bytes, int* S, int* SB) {
  int sb = 0;
  for (int i = 0; i < n; ++i) {
    const int b = stage_layout(geos[i]).bytes;
    sb = b > sb ? b : sb;
  }
  const int avail = kEngineSmemMax - static_bytes - 1024;
  int s = sb > 0 ? avail / sb : 0;
  if (s > kMaxStages) s = kMaxStages;
  *S = s;
  *SB = sb;
}

cudaError_t launch_units(const UnitJob& J, bool f16a, int sms, cudaStream_t st) {
  // the down operand (h) is bf16 hi + lo whatever the activation type
  const bool f = (J.mat & 1) ? false : f16a;
  switch (J.C.geo[J.mat].t.fmt) {
    case MOE_FMT_AFFINE4_G64: return launch_fmt<MOE_FMT_AFFINE4_G64>(J, f, sms, st);
    case MOE_FMT_AFFINE3_G64: return launch_fmt<MOE_FMT_AFFINE3_G64>(J, f, sms, st);
    case MOE_FMT_W4A16_SYM_G128: return launch_fmt<MOE_FMT_W4A16_SYM_G128>(J, f, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_xsum(const uint16_t* x, int T, int H, bool f16, const TileGeo& g13,
                        float* xsum, cudaStream_t st) {
  const int tasks = T * (H >> 7);
  if (tasks <= 0) return cudaSuccess;
  k_xsum<<<(tasks + 7) / 8, 256, 0, st>>>(x, T, H, f16 ? 1 : 0, g13, xsum);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& A, cudaStream_t st) {
  if (A.T <= 0) return cudaSuccess;
  k_combine<<<A.H / kUnitRows, 256, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace moe
