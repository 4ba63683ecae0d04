// decode.cu -- the whole decode layer in one persistent launch.
//
// One CTA per SM, co-resident (cooperative launch), 19 warps each.
//   start    the producer claims its first unit from the grid's queue; the
//            first ceil(T/8) * I/64 queue entries are the shared expert's
//            gate/up units, which need no routing, so a CTA that drew one
//            starts streaming its weight items at once;
//   phase 0  router rows (one k-split of one row per warp) and activation-sum
//            tasks spread over the grid; every logit is published as one
//            64-bit word tagged with the call's generation number, the
//            activation-sum tasks are counted;
//   routing  every CTA polls the tagged logits until all carry this call's
//            generation, then builds the whole routing table itself in shared
//            memory (top-k, bucketing, sub-slots): no fence, no grid-wide
//            counter and no second round trip;
//   phase 1  the item engine (engine.cuh) over the queue: shared gate/up,
//            routed gate/up (sub-slot major), shared down, routed down,
//            combine pieces.  Each producer claims the next queue entry with
//            one atomic as soon as it has published the previous one, so the
//            grid balances itself; a unit waits only on units earlier in the
//            queue (down on its sub-slot's gate/up units, a combine piece on
//            the down units of its rows), which are claimed and never wait
//            on later ones.
// Producers of data never wait: a finished gate/up or down unit adds 1 to a
// counter with a release reduction.  Only the operand warp polls, just
// before it copies operands that other CTAs write (h rows, y rows for the
// combine); weights are fetched ahead regardless.  The arithmetic is the
// standalone kernels' (same device functions), so outputs are identical bit
// for bit.
//
// Every wait is bounded: after the workspace's limit (one second by default)
// it writes MOE_ERR_TIMEOUT to the workspace status word and every later wait
// of the CTA returns at once, so the launch ends (with garbage output; the
// workspace must then be re-initialised).  The last CTA to leave zeroes the
// counters.
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

// Shared-expert gate/up unit v (queue entries 0 .. ceil(T/8) * I/64 - 1):
// decodable before routing.
// Activation-sum tasks of a call (one per token and 128 columns); gate/up
// operands wait until they are all done.
__device__ __forceinline__ int n_xsum_tasks(const DecodeArgs& A) {
  return A.R.T * (A.R.H >> 7);
}

__device__ __forceinline__ UnitInfo shared_gateup_unit(const DecodeArgs& A, int v) {
  const int ngr = A.C.inter / 64;
  const int ss = v / ngr;
  UnitInfo r{};
  r.kind = kItemGateUp;
  r.mat = 2;
  r.e = 0;
  r.blk = v - ss * ngr;
  r.off = kMaxTok * ss;
  r.cnt = min(kMaxTok, A.R.T - kMaxTok * ss);
  r.nch = A.C.geo[2].t.nch;
  r.rows = kRowsDirect;
  r.signal = kSharedReady + ss;
  r.wait_ctr = kCtlXsum;
  r.wait_target = n_xsum_tasks(A);
  return r;
}

__device__ __forceinline__ int n_shared_gateup(const DecodeArgs& A) {
  return A.has_shared ? ((A.R.T + kMaxTok - 1) / kMaxTok) * (A.C.inter / 64) : 0;
}

// The grid's queue, resolved from the CTA's own routing table:
//   [nA shared gate/up][nB routed gate/up][nC shared down][nD routed down]
//   [ncp combine pieces]
// gate/up and down units sub-slot major, so a sub-slot's blocks are claimed
// together; claims come from one atomic counter in the workspace.
struct FusedSched {
  const DecodeArgs* A;
  const RouteTable* RT;
  int T, ngr, nrb, ncp, nss_sh, nss, nA, nB, nC, nD;

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
  }
  __device__ int claim(int) const { return atomicAdd(A->ctrl + kCtlQueue, 1); }
  __device__ bool unit(int j, UnitInfo& r) const {
    r = UnitInfo{};
    if (j < nA) {
      r = shared_gateup_unit(*A, j);
      return true;
    }
    j -= nA;
    if (j < nB) {
      const int ss = j / ngr;
      r.kind = kItemGateUp;
      r.mat = 0;
      r.e = RT->ss_e[ss];
      r.blk = j - ss * ngr;
      r.off = RT->ss_off[ss];
      r.cnt = RT->ss_cnt[ss];
      r.nch = A->C.geo[0].t.nch;
      r.rows = kRowsGather;
      r.signal = kCtlReady + ss;
      r.wait_ctr = kCtlXsum;
      r.wait_target = n_xsum_tasks(*A);
      return true;
    }
    j -= nB;
    if (j < nC + nD) {
      const bool sh = j < nC;
      const int v = sh ? j : j - nC;
      const int ss = v / nrb;
      r.kind = kItemDown;
      r.mat = sh ? 3 : 1;
      r.e = sh ? 0 : RT->ss_e[ss];
      r.blk = v - ss * nrb;
      r.off = sh ? kMaxTok * ss : RT->ss_off[ss];
      r.cnt = sh ? min(kMaxTok, T - kMaxTok * ss) : RT->ss_cnt[ss];
      r.nch = A->C.geo[r.mat].t.nch;
      r.rows = sh ? kRowsDirect : kRowsScatter;
      r.signal = kCtlRb + r.blk;
      r.wait_ctr = (sh ? kSharedReady : kCtlReady) + ss;
      r.wait_target = ngr;
      return true;
    }
    j -= nC + nD;
    if (j < ncp) {
      r.kind = kItemCombine;
      r.blk = j;
      r.signal = -1;
      r.wait_ctr = kCtlRb + j * kCombineRows / kUnitRows;
      r.wait_target = nss + nss_sh;
      return true;
    }
    return false;
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
  __shared__ unsigned s_gen;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  int* ctrl = A.ctrl;
  int* status = ctrl + kCtlStatus;
  const int T = A.R.T, H = A.R.H, NE = A.R.E;
  const bool gate = A.R.gq != nullptr;
  const int E1 = NE + (gate ? 1 : 0);
  // this call's generation number: the tag of its published logits
  if (tid == 0) s_gen = unsigned(*(volatile const int*)(ctrl + kCtlGen)) + 1u;
  engine_init(E, P.S, A.ctrl);
  const EngineMem M{smem, smem + P.nob * P.OB, P.OB, P.nob, P.SB, P.S};
  fence_proxy_async();
  __syncthreads();
  const unsigned gen = s_gen;
  unsigned long long* tagged =
      reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ctrl) + kCtlTaggedOffset);
  const int TS = (NE + 2) & ~1;  // row stride of the tagged logits (even: 16-byte pairs)

  // ---- start: the producer's first claim; a shared-expert gate/up unit
  // (no routing needed) starts streaming its weight items now
  ProducerStart pst{0, 0};
  if (warp == kProducerWarp) {
    int j0 = 0;
    if (lane == 0) j0 = atomicAdd(ctrl + kCtlQueue, 1);
    j0 = __shfl_sync(0xffffffffu, j0, 0);
    pst.j = j0;
    if (j0 < n_shared_gateup(A)) {
      const UnitInfo u = shared_gateup_unit(A, j0);
      pst.issued = min(P.S, u.nch);
      for (int c = 0; c < pst.issued; ++c)
        produce_weights(A.C.geo[u.mat], u, c, M.stages + (size_t)c * M.SB, &E.full[c]);
    }
  }

  // ---- phase 0: router rows and activation sums
  // Router blocks of RPB rows x KS k-splits (one warp each), as few rows per
  // CTA as the grid allows so that each SM streams little of the router; x
  // is read through L2 together with the weights.  Each logit is published
  // as a tagged word (no fence, no counter).  Activation-sum tasks go to the
  // CTAs without router rows and are counted.
  const int KS = A.KS;
  const int RPB = max(1, min(kConsumerWarps / KS, (E1 + G - 1) / G));
  const int nrb_router = (E1 + RPB - 1) / RPB;
  const int nx = n_xsum_tasks(A);
  int done = 0;
  if (warp < kConsumerWarps)
    for (int rb = blockIdx.x; rb < nrb_router; rb += G)
      router_rows_cta(A.R, KS, RPB, rb, RT_part, tagged, TS, gen);
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
  if (lane == 0 && done) red_release_add(ctrl + kCtlXsum, done);

  // ---- routing, redundantly in every CTA, from the tagged logits
  {
    int(*wc)[256] = reinterpret_cast<int(*)[256]>(smem);
    const bool first = blockIdx.x == 0;
    route_table_cta(nullptr, nullptr, T, NE, A.k, first ? A.user_idx : nullptr,
                    first ? A.user_w : nullptr, wc, RT, A.R.round_bf16 != 0, tagged, TS, gen,
                    gate, &E.wc, status);
  }
  fence_proxy_async();  // routing scratch (generic writes) before TMA reuses it
  __syncthreads();

  // ---- phase 1: units through the item engine
  {
    const FusedSched sch(&A, &RT);
    if (warp == kProducerWarp)
      producer_run(A.C, E, M, sch, pst);
    else if (warp == kOperandWarp)
      operand_run(A.C, E, M, sch, ctrl);
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
    if (tid == 0) {
      ctrl[kCtlXsum] = 0;
      ctrl[kCtlQueue] = 0;
      ctrl[kCtlGen] = int(gen);
    }
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
