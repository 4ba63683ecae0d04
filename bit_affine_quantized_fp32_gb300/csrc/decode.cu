// decode.cu -- the whole decode layer in one persistent launch.
//
// One CTA per SM, co-resident (cooperative launch), 18 warps each.
//   phase 0  router tasks (one router row x one k-split, partial sums for all
//            tokens) and activation-sum tasks, spread over every warp of the
//            grid; each finished task adds 1 to a workspace counter;
//   routing  every CTA waits for the counter, then builds the whole routing
//            table itself in shared memory (logits from the partial sums,
//            top-k, bucketing, sub-slots): no second grid-wide round trip;
//   phase 1  gate/up units, then down units, then combine pieces, balanced
//            over the CTAs in closed form (FusedSched), run by the item engine
//            (engine.cuh): the producer warp streams items through TMA stages,
//            16 consumer warps compute, a signal warp publishes results.
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
#include "host.h"

namespace moe {

namespace {

// The units of one CTA, resolved from the CTA's own routing table.  Work is
// balanced in closed form (every CTA computes the same assignment):
//   gate/up units ("big", c1 items each; shared expert first, then routed in
//   sub-slot order) go round-robin: big unit b to CTA b mod G;
//   down units ("small", c2 items each; shared first, then routed in sub-slot
//   order, so early indices depend on early gate/up units) first fill the
//   CTAs that got one big unit fewer, q = ceil(c1/c2) each, spread
//   round-robin over them, then the rest go round-robin over all CTAs;
//   combine pieces (kCombineRows output columns each) go to CTAs G-1, G-2,
//   ... (those with the least work).
// A CTA runs its big units, then its small units, then its combine pieces:
// big units never wait, small units wait only on big units, combine pieces
// only on small units, so every wait is on work that is already queued ahead.
struct FusedSched {
  const DecodeArgs* A;
  const RouteTable* RT;
  int T, ngr, nrb, ncp, nss_sh, nss, nA, nB, nC, nD;
  int G, c, NB, NS, r, q, atot, nb, qa, qb, ne;

  __device__ FusedSched(const DecodeArgs* a, const RouteTable* rt) : A(a), RT(rt) {
    T = A->R.T;
    ngr = A->C.inter / 64;
    nrb = A->C.hidden / kUnitRows;
    ncp = A->C.hidden / kCombineRows;
    nss_sh = A->has_shared ? (T + kMaxTok - 1) / kMaxTok : 0;
    nss = RT->nss;
    nA = nss_sh * ngr;
    nB = nss * ngr;
    nC = nss_sh * nrb;
    nD = nss * nrb;
    G = gridDim.x;
    c = blockIdx.x;
    NB = nA + nB;
    NS = nC + nD;
    const int c1 = A->C.geo[0].t.nch, c2 = A->C.geo[1].t.nch;
    r = NB % G;
    q = r ? (c1 + c2 - 1) / c2 : 0;
    atot = min(NS, (G - r) * q);
    nb = NB / G + (c < r ? 1 : 0);
    // phase-A small units of CTA c: i = k*(G-r) + (c-r), k < q, i < atot
    qa = 0;
    if (c >= r && q > 0 && c - r < atot) qa = min(q, (atot - (c - r) + (G - r) - 1) / (G - r));
    // phase-B small units: i = atot + m*G + c < NS
    qb = NS - atot > c ? (NS - atot - c + G - 1) / G : 0;
    // combine piece e on CTA G-1 - (e mod G)
    const int cc = G - 1 - c;
    ne = ncp > cc ? (ncp - cc + G - 1) / G : 0;
  }
  __device__ int n_units() const { return nb + qa + qb + ne; }
  __device__ UnitInfo unit(int j) const {
    UnitInfo r_{};
    r_.wait_ctr = -1;
    if (j < nb) return big(c + j * G);
    j -= nb;
    if (j < qa) return small(j * (G - r) + (c - r));
    j -= qa;
    if (j < qb) return small(atot + j * G + c);
    j -= qb;
    const int e = (G - 1 - c) + j * G;
    r_.kind = kItemCombine;
    r_.blk = e;
    r_.signal = -1;
    r_.wait_ctr = kCtlRb + e * kCombineRows / kUnitRows;
    r_.wait_target = nss + nss_sh;
    return r_;
  }
  __device__ UnitInfo big(int v) const {
    UnitInfo r_{};
    r_.wait_ctr = -1;
    r_.kind = kItemGateUp;
    if (v < nA) {
      const int ss = v / ngr;
      r_.mat = 2;
      r_.e = 0;
      r_.blk = v - ss * ngr;
      r_.off = kMaxTok * ss;
      r_.cnt = min(kMaxTok, T - kMaxTok * ss);
      r_.nch = A->C.geo[2].t.nch;
      r_.rows = kRowsDirect;
      r_.signal = kSharedReady + ss;
      return r_;
    }
    v -= nA;
    const int ss = v / ngr;
    r_.mat = 0;
    r_.e = RT->ss_e[ss];
    r_.blk = v - ss * ngr;
    r_.off = RT->ss_off[ss];
    r_.cnt = RT->ss_cnt[ss];
    r_.nch = A->C.geo[0].t.nch;
    r_.rows = kRowsGather;
    r_.signal = kCtlReady + ss;
    return r_;
  }
  __device__ UnitInfo small(int v) const {
    UnitInfo r_{};
    r_.kind = kItemDown;
    r_.wait_target = ngr;
    if (v < nC) {
      const int ss = v / nrb;
      r_.mat = 3;
      r_.e = 0;
      r_.blk = v - ss * nrb;
      r_.off = kMaxTok * ss;
      r_.cnt = min(kMaxTok, T - kMaxTok * ss);
      r_.nch = A->C.geo[3].t.nch;
      r_.rows = kRowsDirect;
      r_.signal = kCtlRb + r_.blk;
      r_.wait_ctr = kSharedReady + ss;
      return r_;
    }
    v -= nC;
    const int ss = v / nrb;
    r_.mat = 1;
    r_.e = RT->ss_e[ss];
    r_.blk = v - ss * nrb;
    r_.off = RT->ss_off[ss];
    r_.cnt = RT->ss_cnt[ss];
    r_.nch = A->C.geo[1].t.nch;
    r_.rows = kRowsScatter;
    r_.signal = kCtlRb + r_.blk;
    r_.wait_ctr = kCtlReady + ss;
    return r_;
  }
  __device__ const MatSource& source(int mat) const { return A->src[mat]; }
  __device__ const int* perm() const { return RT->perm; }
  __device__ int topk() const { return A->k; }
  __device__ void combine(int blk) const {
    combine_rows(A->C.tg[1].y, A->C.tg[1].yhalf, RT->w, A->has_shared ? A->C.tg[3].y : nullptr,
                 A->has_shared ? A->C.tg[3].y + A->C.tg[3].yhalf : nullptr,
                 A->has_shared && A->R.gq ? RT->sg : nullptr, A->out, T, A->k, A->C.hidden,
                 A->R.f16 != 0, blk * kCombineRows, kCombineRows, threadIdx.x, kConsumers);
  }
};

template <int FMT, int FMT_SH, bool F16A>
__global__ void __launch_bounds__(kEngineThreads, 1)
    k_decode(const __grid_constant__ DecodeArgs A, const EnginePlan P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ EngineSmem E;
  __shared__ RouteTable RT;
  __shared__ float RT_part[kConsumerWarps * 32];  // router partials [warp][T]
  __shared__ int last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  int* ctrl = A.ctrl;
  int* status = ctrl + kCtlStatus;
  const int T = A.R.T, H = A.R.H, NE = A.R.E;
  const bool gate = A.R.gq != nullptr;
  const int E1 = NE + (gate ? 1 : 0);
  engine_init(E, P.S, A.ctrl);
  const EngineMem M{smem, smem + P.nob * P.OB, P.OB, P.nob, P.SB, P.S};
  fence_proxy_async();
  __syncthreads();

  // ---- phase 0: router rows and activation sums
  // Router blocks of RPB rows x KS k-splits (one warp each, rows finalised in
  // shared memory), as few rows per CTA as the grid allows so that each SM
  // streams little of the router; x is read through L2 together with the
  // weights.  Activation-sum tasks go to the CTAs without router rows.
  const int KS = A.KS;
  const int RPB = max(1, min(kConsumerWarps / KS, (E1 + G - 1) / G));
  const int nrb_router = (E1 + RPB - 1) / RPB;
  const int nx = T * (H >> 7);
  int done = 0;
  for (int rb = blockIdx.x; rb < nrb_router; rb += G) {
    router_rows_cta(A.R, KS, RPB * KS, rb, RT_part, A.R.x, NoPre());
    if (tid == 0) red_release_add(ctrl + kCtlPhase0, 1);
  }
  {
    const int free_ctas = nrb_router < G ? G - nrb_router : G;
    const int first = nrb_router < G ? nrb_router : 0;
    const int me = int(blockIdx.x) - first;
    if (me >= 0) {
      for (int i = me + free_ctas * warp; i < nx; i += free_ctas * (kEngineThreads / 32)) {
        xsum_task(A.R.x, H, A.R.f16 != 0, A.C.geo[0].t, const_cast<float*>(A.src[0].Bsum), i);
        ++done;
      }
    }
  }
  __syncwarp();
  if (lane == 0 && done) red_release_add(ctrl + kCtlPhase0, done);
  const int n_tasks = nrb_router + nx;

  // ---- routing, redundantly in every CTA
  if (tid == 0) wait_counter(ctrl + kCtlPhase0, n_tasks, &E.wc, status);
  __syncthreads();
  {
    int(*wc)[256] = reinterpret_cast<int(*)[256]>(smem);
    const bool first = blockIdx.x == 0;
    route_table_cta(A.R.logits, gate ? A.R.gate_logit : nullptr, T, NE, A.k,
                    first ? A.user_idx : nullptr, first ? A.user_w : nullptr, wc, RT,
                    A.R.round_bf16 != 0);
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
  const cudaError_t e = ensure_dynamic_smem((const void*)k_decode<FMT, FMT_SH, F16A>, smem);
  if (e != cudaSuccess) return e;
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
