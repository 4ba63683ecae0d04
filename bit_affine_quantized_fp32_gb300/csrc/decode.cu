// decode.cu -- the whole decode layer in one persistent launch.
//
// One CTA per SM, co-resident (cooperative launch), 17 warps each.
//   phase 0  router tasks (one router row x one k-split, partial sums for all
//            tokens) and activation-sum tasks, spread over every warp of the
//            grid; each finished task adds 1 to a workspace counter;
//   routing  every CTA waits for the counter, then builds the whole routing
//            table itself in shared memory (logits from the partial sums,
//            top-k, bucketing, sub-slots): no second grid-wide round trip;
//   phase 1  units in one global order -- shared-expert gate/up, routed
//            gate/up, shared down, routed down, combine blocks -- unit u going
//            to CTA (u + 1) mod G, run by the item engine (engine.cuh): the
//            producer warp streams items through TMA stages, 16 consumer warps
//            compute.
// Producers of data never wait: a finished gate/up or down unit adds 1 to a
// counter with a release reduction.  Only the producer warp polls, just
// before it copies operands that other CTAs write (h rows, y rows for the
// combine); weights are fetched ahead regardless.  The arithmetic is the
// standalone kernels' (same device functions), so outputs are identical bit
// for bit.
//
// Every wait is bounded: after about a second it writes MOE_ERR_TIMEOUT to the
// workspace status word and every later wait of the CTA returns at once, so
// the launch ends (with garbage output; the workspace must then be
// re-initialised).  The last CTA to leave zeroes the counters.
//
// Sources: "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803",
// comment "Progress on the 4-bit gate" (routing, grouped experts with a SwiGLU
// epilogue, shared slot, fma combine); "Native server: --backend xpu for
// Nemotron on Intel Arc", update comment (per-row expert reads dominate a
// decode round; a real gain needs expert reads shared across rows).

#include "route.cuh"
#include "decode.h"

namespace moe {

namespace {

// The units of one CTA in the global order, resolved from the CTA's own
// routing table.
struct FusedSched {
  const DecodeArgs* A;
  const RouteTable* RT;
  int T, ngr, nrb, nss_sh, nss, nA, nB, nC, nD, total, u0, nu;

  __device__ FusedSched(const DecodeArgs* a, const RouteTable* rt) : A(a), RT(rt) {
    T = A->R.T;
    ngr = A->C.inter / 64;
    nrb = A->C.hidden / kUnitRows;
    nss_sh = A->has_shared ? (T + kMaxTok - 1) / kMaxTok : 0;
    nss = RT->nss;
    nA = nss_sh * ngr;
    nB = nss * ngr;
    nC = nss_sh * nrb;
    nD = nss * nrb;
    total = nA + nB + nC + nD + nrb;
    const int G = gridDim.x;
    u0 = (blockIdx.x + G - 1) % G;
    nu = total > u0 ? (total - u0 + G - 1) / G : 0;
  }
  __device__ int n_units() const { return nu; }
  __device__ UnitInfo unit(int j) const {
    int v = u0 + j * gridDim.x;
    UnitInfo r{};
    r.wait_ctr = -1;
    if (v < nA) {
      const int ss = v / ngr;
      r.kind = kItemGateUp;
      r.mat = 2;
      r.e = 0;
      r.blk = v - ss * ngr;
      r.off = kMaxTok * ss;
      r.cnt = min(kMaxTok, T - kMaxTok * ss);
      r.nch = A->C.geo[2].t.nch;
      r.rows = kRowsDirect;
      r.signal = kSharedReady + ss;
      return r;
    }
    v -= nA;
    if (v < nB) {
      const int ss = v / ngr;
      r.kind = kItemGateUp;
      r.mat = 0;
      r.e = RT->ss_e[ss];
      r.blk = v - ss * ngr;
      r.off = RT->ss_off[ss];
      r.cnt = RT->ss_cnt[ss];
      r.nch = A->C.geo[0].t.nch;
      r.rows = kRowsGather;
      r.signal = kCtlReady + ss;
      return r;
    }
    v -= nB;
    if (v < nC) {
      const int ss = v / nrb;
      r.kind = kItemDown;
      r.mat = 3;
      r.e = 0;
      r.blk = v - ss * nrb;
      r.off = kMaxTok * ss;
      r.cnt = min(kMaxTok, T - kMaxTok * ss);
      r.nch = A->C.geo[3].t.nch;
      r.rows = kRowsDirect;
      r.signal = kCtlRb + r.blk;
      r.wait_ctr = kSharedReady + ss;
      r.wait_target = ngr;
      return r;
    }
    v -= nC;
    if (v < nD) {
      const int ss = v / nrb;
      r.kind = kItemDown;
      r.mat = 1;
      r.e = RT->ss_e[ss];
      r.blk = v - ss * nrb;
      r.off = RT->ss_off[ss];
      r.cnt = RT->ss_cnt[ss];
      r.nch = A->C.geo[1].t.nch;
      r.rows = kRowsScatter;
      r.signal = kCtlRb + r.blk;
      r.wait_ctr = kCtlReady + ss;
      r.wait_target = ngr;
      return r;
    }
    v -= nD;
    r.kind = kItemCombine;
    r.blk = v;
    r.signal = -1;
    r.wait_ctr = kCtlRb + v;
    r.wait_target = nss + nss_sh;
    return r;
  }
  __device__ const MatSource& source(int mat) const { return A->src[mat]; }
  __device__ const int* perm() const { return RT->perm; }
  __device__ int topk() const { return A->k; }
  __device__ void combine(int blk) const {
    combine_rows(A->y, RT->w, A->has_shared ? A->ysh : nullptr,
                 A->has_shared && A->R.gq ? RT->sg : nullptr, A->out, T, A->k, A->C.hidden,
                 A->R.f16 != 0, blk, threadIdx.x, kConsumers);
  }
};

template <int FMT, bool F16A>
__global__ void __launch_bounds__(kEngineThreads, 1)
    k_decode(const __grid_constant__ DecodeArgs A, int S, int SB) {
  extern __shared__ __align__(128) uint8_t stages[];
  __shared__ EngineSmem E;
  __shared__ RouteTable RT;
  __shared__ __align__(8) uint64_t xbar;
  __shared__ int last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  int* ctrl = A.ctrl;
  int* status = ctrl + kCtlStatus;
  const int T = A.R.T, H = A.R.H, NE = A.R.E;
  const bool gate = A.R.gq != nullptr;
  const int E1 = NE + (gate ? 1 : 0);
  engine_init(E, S);
  if (tid == 0) mbar_init(&xbar, 1);
  fence_proxy_async();
  __syncthreads();

  // ---- phase 0: router partial sums and activation sums
  const uint16_t* xs = A.R.x;
  const int xbytes = T * H * 2;
  if (xbytes <= S * SB) {  // x rows into shared memory for the router tasks
    if (tid == 0) {
      mbar_expect_tx(&xbar, unsigned(xbytes));
      for (int o = 0; o < xbytes; o += 65536)
        bulk_g2s(stages + o, reinterpret_cast<const uint8_t*>(A.R.x) + o,
                 unsigned(min(65536, xbytes - o)), &xbar);
    }
    mbar_wait_bounded(&xbar, 0, &E.skip, status);
    xs = reinterpret_cast<const uint16_t*>(stages);
  }
  const int n_router = E1 * A.KS;
  const int n_tasks = n_router + T * (H >> 7);
  int done = 0;
  for (int i = blockIdx.x + G * warp; i < n_tasks; i += G * (kEngineThreads / 32)) {
    if (i < n_router) {
      const int row = i / A.KS, q = i - row * A.KS;
      router_warp_any(A.R, A.KS, row, q, xs, T, A.part + size_t(q) * T * E1 + row, E1);
    } else {
      xsum_task(A.R.x, H, A.R.f16 != 0, A.C.geo[0].t, const_cast<float*>(A.src[0].Bsum),
                i - n_router);
    }
    ++done;
  }
  __syncwarp();
  if (lane == 0 && done) {
    __threadfence();
    red_release_add(ctrl + kCtlPhase0, done);
  }

  // ---- routing, redundantly in every CTA
  if (tid == 0) wait_counter(ctrl + kCtlPhase0, n_tasks, &E.skip, status);
  __syncthreads();
  {
    float* lg = reinterpret_cast<float*>(stages);
    int(*wc)[256] = reinterpret_cast<int(*)[256]>(stages + align128i((T * NE + T) * 4));
    const bool first = blockIdx.x == 0;
    route_table_cta(A.part, A.KS, E1, A.R.bias, gate, T, NE, A.k, first ? A.user_idx : nullptr,
                    first ? A.user_w : nullptr, lg, wc, RT);
  }
  fence_proxy_async();  // routing scratch (generic writes) before TMA reuses it
  __syncthreads();

  // ---- phase 1: units through the item engine
  {
    const FusedSched sch(&A, &RT);
    if (warp == kProducerWarp)
      producer_run(A.C, E, stages, SB, S, sch, ctrl);
    else
      consumer_run<FMT, F16A>(A.C, E, stages, SB, S, sch, ctrl);
  }

  // ---- exit: the last CTA zeroes the counters for the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int v = atomicAdd(ctrl + kCtlExit, 1);
    last = ((v + 1) % G) == 0;
    if (last) __threadfence();
  }
  __syncthreads();
  if (last) {
    if (tid == 0) ctrl[kCtlPhase0] = 0;
    for (int i = kCtlReady + tid; i < kCtlEnd; i += kEngineThreads) ctrl[i] = 0;
  }
}

template <int FMT, bool F16A>
cudaError_t launch_decode_t(const DecodeArgs& A, int sms, cudaStream_t st) {
  int S = 0, SB = 0, smem = 0;
  decode_smem(A, &S, &SB, &smem);
  if (S < 2) return cudaErrorInvalidValue;
  // raise the dynamic shared-memory limit once per device (not a stream
  // operation, so later calls can be captured in graphs)
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] < smem) {
    e = cudaFuncSetAttribute(k_decode<FMT, F16A>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(sms));
  cfg.blockDim = dim3(kEngineThreads);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode<FMT, F16A>, A, S, SB);
}

template <int FMT>
cudaError_t launch_fmt(const DecodeArgs& A, int sms, cudaStream_t st) {
  return A.R.f16 ? launch_decode_t<FMT, true>(A, sms, st)
                 : launch_decode_t<FMT, false>(A, sms, st);
}

}  // namespace

void decode_smem(const DecodeArgs& A, int* S, int* SB, int* bytes) {
  const TileGeo geos[4] = {A.C.geo[0].t, A.C.geo[1].t, A.C.geo[2].t, A.C.geo[3].t};
  const int stat = int(sizeof(EngineSmem) + sizeof(RouteTable) + 64);
  engine_stages(geos, A.has_shared ? 4 : 2, stat, S, SB);
  // the stage area doubles as routing scratch: logits + 8 x 256 ints
  const int scratch = align128i((A.R.T * A.R.E + A.R.T) * 4) + 8 * 256 * 4;
  if (*S * *SB < scratch) *S = 0;
  *bytes = *S * *SB;
}

cudaError_t launch_decode(const DecodeArgs& A, int fmt, int sms, cudaStream_t st) {
  switch (fmt) {
    case MOE_FMT_AFFINE4_G64: return launch_fmt<MOE_FMT_AFFINE4_G64>(A, sms, st);
    case MOE_FMT_AFFINE3_G64: return launch_fmt<MOE_FMT_AFFINE3_G64>(A, sms, st);
    case MOE_FMT_W4A16_SYM_G128: return launch_fmt<MOE_FMT_W4A16_SYM_G128>(A, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
