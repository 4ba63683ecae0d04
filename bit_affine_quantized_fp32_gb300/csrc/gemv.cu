// gemv.cu -- standalone decode-path expert kernels over the shared units:
// gate/up units (with the SwiGLU epilogue), down units, x preparation and the
// weighted combine.  The fused layer kernel (decode.cu) runs the same device
// functions in the same order per unit, so both paths produce the same bits.
//
// Source: "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803",
// comment "Progress on the 4-bit gate": grouped affine experts with a SwiGLU
// epilogue, decode rows summed in fp32, the slots' fma sum rounded once.

#include "kernels.h"

namespace moe {

namespace {

__device__ __forceinline__ Unit unit_at(const UnitJob& J, int u, int nblk) {
  Unit U;
  const int ss = u / nblk;
  U.down = J.down;
  U.blk = u - ss * nblk;
  U.ss = ss;
  subslot_get(J.ss, ss, U.e, U.off, U.cnt);
  return U;
}

// CTA b takes units b, b + grid, ...; each unit is nch k-chunk items, run
// through a kStages-deep pipeline (codes by TMA bulk copy on a per-stage
// mbarrier, operands by cp.async).
template <int FMT, bool F16A, bool DOWN>
__global__ void __launch_bounds__(kUnitThreads, 1) k_units(const UnitJob J) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ EpiSmem E;
  __shared__ __align__(8) uint64_t bars[kStages];
  const TileGeo& tg = J.g.t;
  const StageLayout L = stage_layout(tg);
  if (threadIdx.x == 0)
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
  fence_proxy_async();
  __syncthreads();
  const int nblk = tg.nblk;
  const int nch = tg.nch;
  const int n_units = subslot_count(J.ss) * nblk;
  const int mine = n_units > int(blockIdx.x) ? (n_units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int n_items = mine * nch;
  auto issue = [&](int k) {
    const Unit U = unit_at(J, blockIdx.x + (k / nch) * gridDim.x, nblk);
    const int c = k % nch;
    uint8_t* st = smem + (k % kStages) * L.bytes;
    stage_weights(J.g, U, c, st, L, &bars[k % kStages]);
    stage_operand_async(tg, c, J.op.rowmap, U.off, U.cnt, J.op.B, J.op.Blo, J.op.Bsum, st, L);
  };
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < n_items) issue(s);
    cp_async_commit();
  }
  unsigned phase = 0;  // bit s: parity of the next completion of stage s
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k = 0; k < n_items; ++k) {
    if (k + kStages - 1 < n_items) issue(k + kStages - 1);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    const int sl = k % kStages;
    const bool landed = mbar_wait(&bars[sl], (phase >> sl) & 1u);
    phase ^= 1u << sl;
    if (__syncthreads_or(!landed)) {
      // give up: report, then wait (bounded) for the copies still in flight
      if (threadIdx.x == 0 && J.status) atomicExch(J.status, int(MOE_ERR_TIMEOUT));
      for (int j = k + 1; j < n_items && j < k + kStages; ++j) {  // items issued so far
        const int sj = j % kStages;
        mbar_wait(&bars[sj], (phase >> sj) & 1u);
        phase ^= 1u << sj;
      }
      break;
    }
    const Unit U = unit_at(J, blockIdx.x + (k / nch) * gridDim.x, nblk);
    const int c = k % nch;
    if (c == 0) acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    compute_pass<FMT, F16A, DOWN>(tg, smem + sl * L.bytes, L, U.cnt, acc);
    if (c == nch - 1) {
      if constexpr (DOWN)
        write_down(J.sink, U, acc);
      else
        swiglu_epilogue(acc, E, U, J.inter, J.hh, J.hl, J.hsum, J.hout);
    }
    __syncthreads();
  }
  cp_async_wait<0>();
}

__global__ void k_xprep(const uint16_t* __restrict__ x, int T, int H, int f16,
                        uint16_t* __restrict__ xperm, float* __restrict__ xsum) {
  const int task = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (task >= T * (H >> 6)) return;
  xprep_task(x, H, f16, xperm, xsum, task);
}

__global__ void __launch_bounds__(kUnitThreads) k_combine(const CombineArgs A) {
  const int t0 = blockIdx.y * 64;
  combine_block(A, blockIdx.x, t0, min(A.T, t0 + 64));
}

template <int FMT, bool F16A, bool DOWN>
cudaError_t launch_units_t(const UnitJob& J, int sms, cudaStream_t st) {
  const int smem = kStages * stage_layout(J.g.t).bytes;
  if (smem > kUnitSmemMax) return cudaErrorInvalidValue;
  // dynamic shared memory above 48 KiB needs an opt-in per device; raise it
  // only when a launch needs more than any earlier one on that device
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] < smem) {
    e = cudaFuncSetAttribute(k_units<FMT, F16A, DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  int blocks = J.max_units < sms ? J.max_units : sms;
  if (blocks < 1) blocks = 1;
  k_units<FMT, F16A, DOWN><<<blocks, kUnitThreads, smem, st>>>(J);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_fmt(const UnitJob& J, bool f16a, int sms, cudaStream_t st) {
  if (J.down) return launch_units_t<FMT, false, true>(J, sms, st);
  return f16a ? launch_units_t<FMT, true, false>(J, sms, st)
              : launch_units_t<FMT, false, false>(J, sms, st);
}

}  // namespace

cudaError_t launch_units(const UnitJob& J, bool f16a, int sms, cudaStream_t st) {
  switch (J.g.t.fmt) {
    case MOE_FMT_AFFINE4_G64: return launch_fmt<MOE_FMT_AFFINE4_G64>(J, f16a, sms, st);
    case MOE_FMT_AFFINE3_G64: return launch_fmt<MOE_FMT_AFFINE3_G64>(J, f16a, sms, st);
    case MOE_FMT_W4A16_SYM_G128: return launch_fmt<MOE_FMT_W4A16_SYM_G128>(J, f16a, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_xprep(const uint16_t* x, int T, int H, bool f16, uint16_t* xperm, float* xsum,
                         cudaStream_t st) {
  const long warps = long(T) * (H / 64);
  if (warps == 0) return cudaSuccess;
  k_xprep<<<int((warps + 7) / 8), 256, 0, st>>>(x, T, H, f16 ? 1 : 0, xperm, xsum);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& A, cudaStream_t st) {
  if (A.T <= 0) return cudaSuccess;
  dim3 grid(A.H / kUnitRows, (A.T + 63) / 64);
  k_combine<<<grid, kUnitThreads, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace moe
