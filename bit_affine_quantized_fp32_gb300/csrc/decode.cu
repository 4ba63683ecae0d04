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
    combine_rows(A->C.tg[1].y, A->C.tg[1].yhalf, RT->w, A->has_shared ? A->C.tg[3].y : nullptr,
                 A->has_shared ? A->C.tg[3].y + A->C.tg[3].yhalf : nullptr,
                 A->has_shared && A->R.gq ? RT->sg : nullptr, A->out, T, A->k, A->C.hidden,
                 A->R.f16 != 0, blk, threadIdx.x, kConsumers);
  }
};

template <int FMT, int FMT_SH, bool F16A>
__global__ void __launch_bounds__(kEngineThreads, 1)
    k_decode(const __grid_constant__ DecodeArgs A, const EnginePlan P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ EngineSmem E;
  __shared__ RouteTable RT;
  __shared__ float RT_part[kConsumerWarps * 32];  // router partials [warp][T]
  __shared__ __align__(8) uint64_t xbar;
  __shared__ int last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  int* ctrl = A.ctrl;
  int* status = ctrl + kCtlStatus;
  const int T = A.R.T, H = A.R.H, NE = A.R.E;
  const bool gate = A.R.gq != nullptr;
  const int E1 = NE + (gate ? 1 : 0);
  engine_init(E, P.S);
  const EngineMem M{smem, smem + P.nob * P.OB, P.OB, P.nob, P.SB, P.S};
  if (tid == 0) mbar_init(&xbar, 1);
  fence_proxy_async();
  __syncthreads();

  // ---- phase 0: router partial sums and activation sums
  const int xbytes = T * H * 2;
  // x rows into shared memory for the router blocks of this CTA
  const bool xsm = int(blockIdx.x) < (E1 + kConsumerWarps / A.KS - 1) / (kConsumerWarps / A.KS) &&
                   xbytes <= P.nob * P.OB + P.S * P.SB;
  if (xsm && tid == 0) {
    mbar_expect_tx(&xbar, unsigned(xbytes));
    for (int o = 0; o < xbytes; o += 65536)
      bulk_g2s(smem + o, reinterpret_cast<const uint8_t*>(A.R.x) + o,
               unsigned(min(65536, xbytes - o)), &xbar);
  }
  const uint16_t* xs = xsm ? reinterpret_cast<const uint16_t*>(smem) : A.R.x;
  bool xready = !xsm;
  auto wait_x = [&]() {
    if (!xready) {
      mbar_wait_bounded(&xbar, 0, &E.skip, status);
      xready = true;
    }
  };
  // router blocks (all warps of a CTA, rows finalised in shared memory) first,
  // activation-sum tasks on the CTAs after them
  const int RPB = kConsumerWarps / A.KS;
  const int nrb_router = (E1 + RPB - 1) / RPB;
  const int nx = T * (H >> 7);
  int done = 0;
  for (int rb = blockIdx.x; rb < nrb_router; rb += G) {
    router_rows_cta(A.R, A.KS, kConsumerWarps, rb, RT_part, xs, wait_x);
    if (tid == 0) red_release_add(ctrl + kCtlPhase0, 1);
  }
  const int xb = (blockIdx.x + G - nrb_router % G) % G;
  for (int i = xb + G * warp; i < nx; i += G * (kEngineThreads / 32)) {
    xsum_task(A.R.x, H, A.R.f16 != 0, A.C.geo[0].t, const_cast<float*>(A.src[0].Bsum), i);
    ++done;
  }
  wait_x();  // every thread: the copy has landed before the shared memory is reused
  __syncwarp();
  if (lane == 0 && done) red_release_add(ctrl + kCtlPhase0, done);
  const int n_tasks = nrb_router + nx;

  // ---- routing, redundantly in every CTA
  if (tid == 0) wait_counter(ctrl + kCtlPhase0, n_tasks, &E.skip, status);
  __syncthreads();
  {
    int(*wc)[256] = reinterpret_cast<int(*)[256]>(smem);
    const bool first = blockIdx.x == 0;
    route_table_cta(A.R.logits, gate ? A.R.gate_logit : nullptr, T, NE, A.k,
                    first ? A.user_idx : nullptr, first ? A.user_w : nullptr, wc, RT);
  }
  fence_proxy_async();  // routing scratch (generic writes) before TMA reuses it
  __syncthreads();

  // ---- phase 1: units through the item engine
  {
    const FusedSched sch(&A, &RT);
    if (warp == kProducerWarp)
      producer_run(A.C, E, M, sch, ctrl);
    else if (warp == kSignalWarp)
      signal_run(E, sch, ctrl, status);
    else
      consumer_run<FMT, FMT_SH, F16A>(A.C, E, M, sch);
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

template <int FMT, int FMT_SH, bool F16A>
cudaError_t launch_decode_t(const DecodeArgs& A, int sms, cudaStream_t st) {
  const EnginePlan P = decode_plan(A);
  if (P.S < 2) return cudaErrorInvalidValue;
  const int smem = P.bytes();
  // raise the dynamic shared-memory limit once per device (not a stream
  // operation, so later calls can be captured in graphs)
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] < smem) {
    e = cudaFuncSetAttribute(k_decode<FMT, FMT_SH, F16A>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
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
  return cudaLaunchKernelEx(&cfg, k_decode<FMT, FMT_SH, F16A>, A, P);
}

template <int FMT, int FMT_SH>
cudaError_t launch_fmt2(const DecodeArgs& A, int sms, cudaStream_t st) {
  return A.R.f16 ? launch_decode_t<FMT, FMT_SH, true>(A, sms, st)
                 : launch_decode_t<FMT, FMT_SH, false>(A, sms, st);
}

template <int FMT>
cudaError_t launch_fmt(const DecodeArgs& A, int fmt_sh, int sms, cudaStream_t st) {
  switch (fmt_sh) {
    case MOE_FMT_AFFINE4_G64: return launch_fmt2<FMT, MOE_FMT_AFFINE4_G64>(A, sms, st);
    case MOE_FMT_AFFINE3_G64: return launch_fmt2<FMT, MOE_FMT_AFFINE3_G64>(A, sms, st);
    case MOE_FMT_W4A16_SYM_G128: return launch_fmt2<FMT, MOE_FMT_W4A16_SYM_G128>(A, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

EnginePlan decode_plan(const DecodeArgs& A) {
  const TileGeo geos[4] = {A.C.geo[0].t, A.C.geo[1].t, A.C.geo[2].t, A.C.geo[3].t};
  const int stat = int(sizeof(EngineSmem) + sizeof(RouteTable) + 64);
  EnginePlan P = engine_plan(geos, A.has_shared ? 4 : 2, stat);
  // the dynamic area doubles as routing scratch (8 x 256 ints)
  if (P.bytes() < 8 * 256 * 4) P.S = 0;
  return P;
}

cudaError_t launch_decode(const DecodeArgs& A, int fmt, int fmt_sh, int sms, cudaStream_t st) {
  switch (fmt) {
    case MOE_FMT_AFFINE4_G64: return launch_fmt<MOE_FMT_AFFINE4_G64>(A, fmt_sh, sms, st);
    case MOE_FMT_AFFINE3_G64: return launch_fmt<MOE_FMT_AFFINE3_G64>(A, fmt_sh, sms, st);
    case MOE_FMT_W4A16_SYM_G128: return launch_fmt<MOE_FMT_W4A16_SYM_G128>(A, fmt_sh, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
