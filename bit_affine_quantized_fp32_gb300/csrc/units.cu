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
#include "host.h"

namespace moe {

namespace {

__device__ __forceinline__ int subslot_count(const SubSlots& S) {
  return S.n ? __ldcg(S.n) : (S.fixed_T + kMaxTok - 1) / kMaxTok;
}

// The units of this CTA: claims n = 0, 1, ... are queue indices
// blockIdx.x + n * gridDim.x over n_subslots x blocks, sub-slot major.
struct JobSched {
  const UnitJob* J;
  int nblk, total;
  __device__ explicit JobSched(const UnitJob* j) : J(j) {
    nblk = J->C.geo[J->mat].t.nblk;
    total = subslot_count(J->ss) * nblk;
  }
  __device__ int claim(int n) const { return blockIdx.x + n * gridDim.x; }
  __device__ bool unit(int u, UnitInfo& r) const {
    r = UnitInfo{};
    if (u >= total) return false;
    const int ss = u / nblk;
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
    return true;
  }
  __device__ const MatSource& source(int) const { return J->src; }
  __device__ const int* perm() const { return J->perm; }
  __device__ int topk() const { return J->k; }
  __device__ void combine(int) const {}
};

template <int FMT, bool F16A>
__global__ void __launch_bounds__(kEngineThreads, 1)
    k_units(const __grid_constant__ UnitJob J, const EnginePlan P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ EngineSmem E;
  engine_init(E, P.S, J.C.status);
  fence_proxy_async();
  __syncthreads();
  const EngineMem M{smem, smem + P.nob * P.OB, P.OB, P.nob, P.SB, P.S};
  const JobSched sch(&J);
  const int warp = threadIdx.x >> 5;
  if (warp == kProducerWarp)
    producer_run(J.C, E, M, sch, ProducerStart{sch.claim(0), 0});
  else if (warp == kOperandWarp)
    operand_run(J.C, E, M, sch, nullptr);
  else if (warp == kSignalWarp)
    signal_run(E, sch, nullptr, J.C.status);  // reads the ring; nothing to publish
  else
    consumer_run<FMT, FMT, F16A>(J.C, E, M, sch);
}

__global__ void k_xsum(const uint16_t* __restrict__ x, int T, int H, int f16, TileGeo g13,
                       float* __restrict__ xsum) {
  const int task = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (task >= T * (H >> 7)) return;
  xsum_task(x, H, f16 != 0, g13, xsum, task);
}

// xsum_task over bf16 activations plus their fp16 copy (exact in fp16's
// normal range; a value beyond it sets MOE_ERR_RANGE): lane l of the warp of
// (token, 128 columns) converts the 4 columns it sums.
__global__ void k_xsum_f16(const uint16_t* __restrict__ x, int T, int H, TileGeo g13,
                           float* __restrict__ xsum, uint16_t* __restrict__ xh, int* status) {
  const int task = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (task >= T * (H >> 7)) return;
  xsum_task(x, H, false, g13, xsum, task);
  const int lane = threadIdx.x & 31, nb = H >> 7;
  const int t = task / nb, q = task - t * nb;
  const size_t at = (size_t)t * H + q * 128 + 4 * lane;
  const uint2 v = *reinterpret_cast<const uint2*>(x + at);
  const float f0 = __uint_as_float(v.x << 16), f1 = __uint_as_float(v.x & 0xFFFF0000u);
  const float f2 = __uint_as_float(v.y << 16), f3 = __uint_as_float(v.y & 0xFFFF0000u);
  const __half2 h01 = __floats2half2_rn(f0, f1), h23 = __floats2half2_rn(f2, f3);
  *reinterpret_cast<uint2*>(xh + at) = make_uint2(*reinterpret_cast<const uint32_t*>(&h01),
                                                  *reinterpret_cast<const uint32_t*>(&h23));
  if (!(fabsf(f0) <= 65504.f) || !(fabsf(f1) <= 65504.f) || !(fabsf(f2) <= 65504.f) ||
      !(fabsf(f3) <= 65504.f))
    atomicExch(status, int(MOE_ERR_RANGE));
}

// The combine of combine_rows, element for element the same arithmetic, laid
// out for streaming: a block takes kCmbTok tokens x kCmbCols columns; the
// tokens' slot weights (bf16-rounded in the chain), the second-plane flags and
// the shared weights are read once into shared memory, then each thread reads
// four consecutive columns of every slot row with 16-byte loads.
constexpr int kCmbTok = 4, kCmbCols = 512, kCmbThreads = kCmbCols / 4;
__global__ void __launch_bounds__(kCmbThreads) k_combine(const CombineArgs A) {
  __shared__ float sw[kCmbTok][kMaxTopK];
  __shared__ int stwo[kCmbTok][kMaxTopK];
  __shared__ float ssg[kCmbTok];
  const int t0 = blockIdx.y * kCmbTok;
  const int Tn = min(kCmbTok, A.T - t0);
  const int tid = threadIdx.x;
  const bool rb = A.round_bf16 != 0;
  if (tid < kCmbTok * kMaxTopK) {
    const int tt = tid / kMaxTopK, j = tid - tt * kMaxTopK;
    float wv = 0.f;
    int two = 0;
    if (tt < Tn && j < A.k) {
      const int t = t0 + tt;
      wv = A.w[t * A.k + j];
      if (rb) wv = round_bf16(wv);
      two = A.yhalf != 0;
      if (two && A.idx) {
        const int e = __ldg(A.idx + t * A.k + j);
        two = __ldg(A.offsets + e + 1) - __ldg(A.offsets + e) <= A.one_plane_max;
      }
    }
    sw[tt][j] = wv;
    stwo[tt][j] = two;
  }
  if (tid < kCmbTok) {
    float v = 1.f;
    if (A.sg && tid < Tn) v = rb ? round_bf16(A.sg[t0 + tid]) : A.sg[t0 + tid];
    ssg[tid] = v;
  }
  __syncthreads();
  const int h = blockIdx.x * kCmbCols + 4 * tid;
  if (h >= A.H) return;
  for (int tt = 0; tt < Tn; ++tt) {
    const int t = t0 + tt;
    float4 ya[kMaxTopK], yb[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < A.k) {
        const size_t a = (size_t)(t * A.k + j) * A.H + h;
        ya[j] = __ldcg(reinterpret_cast<const float4*>(A.y + a));
        yb[j] = stwo[tt][j] ? __ldcg(reinterpret_cast<const float4*>(A.y + A.yhalf + a))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float4 vs = make_float4(0.f, 0.f, 0.f, 0.f);
    if (A.ysh) {
      const size_t a = (size_t)t * A.H + h;
      vs = __ldcg(reinterpret_cast<const float4*>(A.ysh + a));
      if (A.ysh2) {
        const float4 v2 = __ldcg(reinterpret_cast<const float4*>(A.ysh2 + a));
        vs = make_float4(vs.x + v2.x, vs.y + v2.y, vs.z + v2.z, vs.w + v2.w);
      }
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < A.k) {
        const float wj = sw[tt][j];
        const float y4[4] = {ya[j].x, ya[j].y, ya[j].z, ya[j].w};
        const float b4[4] = {yb[j].x, yb[j].y, yb[j].z, yb[j].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = fmaf(wj, A.yhalf ? y4[c] + b4[c] : y4[c], acc[c]);
      }
    if (A.ysh) {
      const float v4[4] = {vs.x, vs.y, vs.z, vs.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] = fmaf(ssg[tt], v4[c], acc[c]);
    }
    const bool f16 = A.f16 != 0;
    const uint32_t lo = uint32_t(float_to_act_bits(acc[0], f16)) |
                        (uint32_t(float_to_act_bits(acc[1], f16)) << 16);
    const uint32_t hi = uint32_t(float_to_act_bits(acc[2], f16)) |
                        (uint32_t(float_to_act_bits(acc[3], f16)) << 16);
    *reinterpret_cast<uint2*>(A.out + (size_t)t * A.H + h) = make_uint2(lo, hi);
  }
}

// dst = a + b elementwise (the two k-half planes of a down projection)
__global__ void k_add_planes(const float* __restrict__ a, const float* __restrict__ b,
                             float* __restrict__ dst, long n) {
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = a[i] + b[i];
}

__global__ void k_store_word(int* p, int v) { *p = v; }

template <int FMT, bool F16A>
cudaError_t launch_units_t(const UnitJob& J, int sms, cudaStream_t st) {
  const TileGeo geos[1] = {J.C.geo[J.mat].t};
  const EnginePlan P = engine_plan(geos, 1, int(sizeof(EngineSmem)));
  if (P.S < 2) return cudaErrorInvalidValue;
  const int smem = P.bytes();
  const cudaError_t e = ensure_dynamic_smem((const void*)k_units<FMT, F16A>, smem);
  if (e != cudaSuccess) return e;
  const int grid = J.max_units < sms ? J.max_units : sms;
  if (grid <= 0) return cudaSuccess;
  k_units<FMT, F16A><<<grid, kEngineThreads, smem, st>>>(J, P);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_fmt(const UnitJob& J, bool f16a, int sms, cudaStream_t st) {
  return f16a ? launch_units_t<FMT, true>(J, sms, st) : launch_units_t<FMT, false>(J, sms, st);
}

}  // namespace

EnginePlan engine_plan(const TileGeo* geos, int n, int static_bytes) {
  EnginePlan P{0, 2, 0, 0};
  for (int i = 0; i < n; ++i) {
    const int sb = stage_bytes(geos[i]), ob = op_layout(geos[i]).bytes;
    P.SB = sb > P.SB ? sb : P.SB;
    P.OB = ob > P.OB ? ob : P.OB;
  }
  const int avail = kEngineSmemMax - static_bytes - 1024;
  if (P.SB <= 0) return P;
  P.S = (avail - 2 * P.OB) / P.SB;
  if (P.S < 2) {
    P.nob = 1;
    P.S = (avail - P.OB) / P.SB;
  }
  if (P.S > kMaxStages) P.S = kMaxStages;
  if (P.S < 0) P.S = 0;
  return P;
}

cudaError_t launch_units(const UnitJob& J, bool f16a, int sms, cudaStream_t st) {
  // the down operand (h) is bf16 hi + lo whatever the activation type
  const bool f = (J.mat & 1) ? false : f16a;
  switch (J.C.geo[J.mat].t.fmt) {
    case MOE_FMT_AFFINE4_G64: return launch_fmt<MOE_FMT_AFFINE4_G64>(J, f, sms, st);
    case MOE_FMT_AFFINE3_G64: return launch_fmt<MOE_FMT_AFFINE3_G64>(J, f, sms, st);
    case MOE_FMT_W4A16_SYM_G128: return launch_fmt<MOE_FMT_W4A16_SYM_G128>(J, f, sms, st);
    case MOE_FMT_AFFINE2_G64: return launch_fmt<MOE_FMT_AFFINE2_G64>(J, f, sms, st);
    case MOE_FMT_AFFINE5_G64: return launch_fmt<MOE_FMT_AFFINE5_G64>(J, f, sms, st);
    case MOE_FMT_AFFINE6_G64: return launch_fmt<MOE_FMT_AFFINE6_G64>(J, f, sms, st);
    case MOE_FMT_AFFINE8_G64: return launch_fmt<MOE_FMT_AFFINE8_G64>(J, f, sms, st);
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

cudaError_t launch_xsum_f16(const uint16_t* x, int T, int H, const TileGeo& g13, float* xsum,
                            uint16_t* xh, int* status, cudaStream_t st) {
  const int tasks = T * (H >> 7);
  if (tasks <= 0) return cudaSuccess;
  k_xsum_f16<<<(tasks + 7) / 8, 256, 0, st>>>(x, T, H, g13, xsum, xh, status);
  return cudaGetLastError();
}

cudaError_t launch_add_planes(const float* a, const float* b, float* dst, long n,
                              cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  k_add_planes<<<unsigned((n + 255) / 256), 256, 0, st>>>(a, b, dst, n);
  return cudaGetLastError();
}

cudaError_t launch_store_word(int* p, int v, cudaStream_t st) {
  k_store_word<<<1, 1, 0, st>>>(p, v);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& A, cudaStream_t st) {
  if (A.T <= 0) return cudaSuccess;
  k_combine<<<dim3((A.H + kCmbCols - 1) / kCmbCols, (A.T + kCmbTok - 1) / kCmbTok), kCmbThreads, 0,
              st>>>(A);
  return cudaGetLastError();
}

}  // namespace moe
