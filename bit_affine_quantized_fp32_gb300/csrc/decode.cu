// decode.cu -- the whole decode layer in one persistent launch.
//
// One CTA per SM, co-resident (cooperative launch).  Work is scheduled
// statically, so no CTA ever waits to be told what to do:
//   phase 0  router blocks and x-preparation blocks, spread over the CTAs;
//            CTA 0 then waits for the logits and does top-k, weights,
//            bucketing and the sub-slot table, and raises the routing flag;
//   phase 1  units in one global order -- shared-expert gate/up, routed
//            gate/up, shared down, routed down -- unit u going to CTA
//            (u + 1) mod G, streamed as k-chunk items through a 3-stage
//            pipeline (weights by TMA bulk copies, operands by cp.async);
//   phase 2  the weighted combine of each 128-row output block.
// Producers never wait: a finished gate/up unit, down unit or phase-0 block
// adds 1 to a workspace counter with a release reduction.  Consumers poll
// only where data is needed: a down unit's operand rows (h) are copied once
// all 64-row groups of its sub-slot are counted, a combine block once all down
// units of that block are.  Down-unit weights are fetched early regardless.
// The arithmetic is the standalone kernels' (units.cuh, route.cuh), so the
// outputs are identical bit for bit.
//
// Every wait is bounded: after about a second it writes MOE_ERR_TIMEOUT to the
// workspace status word, drains its copies and returns (the workspace must
// then be re-initialised).  The last CTA to leave zeroes the counters.
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

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait (one thread): true once *p >= target; false after the limit,
// with the workspace status set to MOE_ERR_TIMEOUT.
__device__ __noinline__ bool wait_geq(const int* p, int target, int* status) {
  unsigned ns = 32;
  for (int i = 0; i < (1 << 21); ++i) {
    if (ld_acquire(p) >= target) return true;
    __nanosleep(ns);
    if (ns < 512) ns <<= 1;
  }
  atomicExch(status, int(MOE_ERR_TIMEOUT));
  return false;
}

enum : int { kSegA = 0, kSegB, kSegC, kSegD, kSegE, kSegEnd };

struct CtaState {
  float part[8 * kRouterTT];
  int wcount[8];
  int tab_e[kMaxSubFused];
  int tab_off[kMaxSubFused];
  int tab_cnt[kMaxSubFused];
  int tab_rows[kMaxSubFused][kMaxTok];
  int n_ss;
  int flag;
};

// Where unit index u stands in the global order (uniform over the CTA).
struct Resolved {
  int seg;
  Unit U;
  int nch;
};

struct Sched {
  int T, ngr, nrb, nss_sh, nA, nss;
  __device__ int nB() const { return nss * ngr; }
  __device__ int nC() const { return nss_sh * nrb; }
  __device__ int nD() const { return nss * nrb; }
};

__device__ __forceinline__ Resolved resolve(const DecodeArgs& A, const CtaState& S,
                                            const Sched& Q, int u) {
  Resolved r{};
  if (u < Q.nA) {
    const int ss = u / Q.ngr;
    r.seg = kSegA;
    r.U = Unit{0, 0, u - ss * Q.ngr, kMaxTok * ss, min(kMaxTok, Q.T - kMaxTok * ss), ss};
    r.nch = A.g13s.t.nch;
    return r;
  }
  int v = u - Q.nA;
  if (v < Q.nB()) {
    const int ss = v / Q.ngr;
    r.seg = kSegB;
    r.U = Unit{0, S.tab_e[ss], v - ss * Q.ngr, S.tab_off[ss], S.tab_cnt[ss], ss};
    r.nch = A.g13.t.nch;
    return r;
  }
  v -= Q.nB();
  if (v < Q.nC()) {
    const int ss = v / Q.nrb;
    r.seg = kSegC;
    r.U = Unit{1, 0, v - ss * Q.nrb, kMaxTok * ss, min(kMaxTok, Q.T - kMaxTok * ss), ss};
    r.nch = A.g2s.t.nch;
    return r;
  }
  v -= Q.nC();
  if (v < Q.nD()) {
    const int ss = v / Q.nrb;
    r.seg = kSegD;
    r.U = Unit{1, S.tab_e[ss], v - ss * Q.nrb, S.tab_off[ss], S.tab_cnt[ss], ss};
    r.nch = A.g2.t.nch;
    return r;
  }
  v -= Q.nD();
  r.seg = v < Q.nrb ? kSegE : kSegEnd;
  r.U = Unit{0, 0, v, 0, 0, 0};
  r.nch = 0;
  return r;
}

__device__ __forceinline__ const MatGeo& geo_of(const DecodeArgs& A, int seg) {
  return seg == kSegA ? A.g13s : seg == kSegB ? A.g13 : seg == kSegC ? A.g2s : A.g2;
}

__device__ __forceinline__ OperandSrc op_of(const DecodeArgs& A, int seg) {
  switch (seg) {
    case kSegA: return OperandSrc{A.xperm, nullptr, A.xsum, nullptr};
    case kSegB: return OperandSrc{A.xperm, nullptr, A.xsum, nullptr};  // rows: sub-slot table
    case kSegC: return OperandSrc{A.sh_hh, A.sh_hl, A.sh_hsum, nullptr};
    default: return OperandSrc{A.hh, A.hl, A.hsum, nullptr};
  }
}

// Counter that says the operand rows (h) of a down unit are complete.
__device__ __forceinline__ int* ready_ctr(const DecodeArgs& A, int seg, int ss) {
  return A.ctrl + (seg == kSegC || seg == kSegA ? kSharedReady : kCtlReady) + ss;
}

// Top-k, weights, bucketing and the sub-slot table by one CTA (all in shared
// memory), then the routing flag.
__device__ void do_routing(const DecodeArgs& A, uint8_t* smem) {
  route_small_cta(A.R.logits, A.R.gq ? A.R.gate_logit : nullptr, A.R.T, A.R.E, A.k, A.idx, A.w,
                  A.sgw, A.user_idx, A.user_w, A.offsets, A.perm, A.nss, A.se, A.so, A.sc,
                  A.rows, *reinterpret_cast<SmallRouteSmem*>(smem));
  if (threadIdx.x == 0) {
    __threadfence();
    st_release(A.ctrl + kCtlRoutingReady, 1);
  }
  __syncthreads();
}

template <bool F16A>
__device__ __forceinline__ void compute_any(const TileGeo& g, int down, const uint8_t* st,
                                            const StageLayout& L, int ntok, float (&acc)[4]) {
  if (down) {
    if (g.fmt == MOE_FMT_AFFINE4_G64)
      compute_pass<MOE_FMT_AFFINE4_G64, false, true>(g, st, L, ntok, acc);
    else if (g.fmt == MOE_FMT_AFFINE3_G64)
      compute_pass<MOE_FMT_AFFINE3_G64, false, true>(g, st, L, ntok, acc);
    else
      compute_pass<MOE_FMT_W4A16_SYM_G128, false, true>(g, st, L, ntok, acc);
  } else {
    if (g.fmt == MOE_FMT_AFFINE4_G64)
      compute_pass<MOE_FMT_AFFINE4_G64, F16A, false>(g, st, L, ntok, acc);
    else if (g.fmt == MOE_FMT_AFFINE3_G64)
      compute_pass<MOE_FMT_AFFINE3_G64, F16A, false>(g, st, L, ntok, acc);
    else
      compute_pass<MOE_FMT_W4A16_SYM_G128, F16A, false>(g, st, L, ntok, acc);
  }
}

template <bool F16A>
__global__ void __launch_bounds__(kUnitThreads, 1) k_decode(const DecodeArgs A, int SB) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ CtaState S;
  __shared__ EpiSmem Ep;
  __shared__ __align__(8) uint64_t bars[kStages];
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0)
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
  const int G = gridDim.x;
  int* ctrl = A.ctrl;
  int* status = ctrl + kCtlStatus;
  const int T = A.R.T, H = A.R.H, I = A.inter;

  // ---- phase 0: router blocks, x preparation, then routing on CTA 0
  const int ntask = T * (H / 64);
  // x rows in shared memory for the router blocks (when they fit)
  const uint16_t* xs = A.R.x;
  if (int(blockIdx.x) < A.NR && T * H * 2 <= kStages * SB) {
    const int n16 = T * H * 2 / 16;
    for (int i = tid; i < n16; i += kUnitThreads)
      cp_async16(smem + 16 * i, reinterpret_cast<const uint8_t*>(A.R.x) + 16 * i);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    xs = reinterpret_cast<const uint16_t*>(smem);
  }
  for (int w = blockIdx.x; w < A.NR + A.XB; w += G) {
    if (w < A.NR) {
      router_block_any(A.R, A.KS, w, S.part, xs, 0, T);
    } else {
      const int task = (w - A.NR) * kUnitWarps + warp;
      if (task < ntask) xprep_task(A.R.x, H, A.f16, A.xperm, A.xsum, task);
      __syncthreads();
    }
    if (tid == 0) {
      __threadfence();
      red_release_add(ctrl + (w < A.NR ? kCtlRouterDone : kCtlXprepDone), 1);
    }
  }
  if (blockIdx.x == 0) {
    if (tid == 0) S.flag = wait_geq(ctrl + kCtlRouterDone, A.NR, status);
    __syncthreads();
    if (!S.flag) return;
    do_routing(A, smem);
  }
  if (tid == 0) S.flag = wait_geq(ctrl + kCtlXprepDone, A.XB, status);
  fence_proxy_async();  // barrier inits and phase-0 shared-memory writes before TMA
  __syncthreads();
  if (!S.flag) return;

  // ---- phase 1: units
  Sched Q;
  Q.T = T;
  Q.ngr = I / 64;
  Q.nrb = H / kUnitRows;
  Q.nss_sh = A.has_shared ? (T + kMaxTok - 1) / kMaxTok : 0;
  Q.nA = Q.nss_sh * Q.ngr;
  Q.nss = 0;
  bool routed = false;
  bool aborted = false;
  // resolve unit j of this CTA (uniform; waits for the routing table once)
  const int u0 = (blockIdx.x + G - 1) % G;
  auto load = [&](int j, Resolved& r) -> bool {
    const int u = u0 + j * G;
    if (u >= Q.nA && !routed) {
      if (tid == 0) S.flag = wait_geq(ctrl + kCtlRoutingReady, 1, status);
      __syncthreads();
      if (!S.flag) return false;
      const int n = __ldcg(A.nss);
      for (int i = tid; i < n; i += kUnitThreads) {
        S.tab_e[i] = __ldcg(A.se + i);
        S.tab_off[i] = __ldcg(A.so + i);
        S.tab_cnt[i] = __ldcg(A.sc + i);
      }
      for (int i = tid; i < n * kMaxTok; i += kUnitThreads)
        S.tab_rows[i / kMaxTok][i % kMaxTok] = __ldcg(A.rows + i);
      __syncthreads();
      Q.nss = n;
      routed = true;
    }
    r = resolve(A, S, Q, u);
    return true;
  };
  unsigned phase = 0;     // bit s: parity of the next completion of stage s
  unsigned inflight = 0;  // bit s: stage s has copies not yet waited for
  auto issue_weights = [&](const Resolved& r, int c, int slot) {
    const MatGeo& g = geo_of(A, r.seg);
    stage_weights(g, r.U, c, smem + slot * SB, stage_layout(g.t), &bars[slot]);
    inflight |= 1u << slot;
  };
  auto drain = [&]() {  // bounded wait for every stage still being filled
    for (int sj = 0; sj < kStages; ++sj)
      if (inflight & (1u << sj)) {
        mbar_wait(&bars[sj], (phase >> sj) & 1u);
        phase ^= 1u << sj;
      }
    inflight = 0;
  };
  auto issue_operand = [&](const Resolved& r, int c, int slot, bool ready, unsigned& defer) {
    if (!ready) {
      defer |= 1u << slot;
      return;
    }
    const MatGeo& g = geo_of(A, r.seg);
    const OperandSrc op = op_of(A, r.seg);
    if (r.seg == kSegB)
      stage_operand_async(g.t, c, S.tab_rows[r.U.ss], 0, r.U.cnt, op.B, op.Blo, op.Bsum,
                          smem + slot * SB, stage_layout(g.t));
    else
      stage_operand_async(g.t, c, nullptr, r.U.off, r.U.cnt, op.B, op.Blo, op.Bsum,
                          smem + slot * SB, stage_layout(g.t));
  };
  auto is_ready = [&](const Resolved& r) -> bool {
    return !r.U.down || ld_acquire(ready_ctr(A, r.seg, r.U.ss)) >= Q.ngr;
  };

  int ij = 0, ic = 0;
  Resolved ir;
  unsigned defer = 0;
  if (!load(0, ir)) return;
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (ir.seg <= kSegD) {
      issue_weights(ir, ic, s);
      issue_operand(ir, ic, s, is_ready(ir), defer);
    }
    cp_async_commit();
    if (ir.seg <= kSegD && ++ic >= ir.nch) {
      ic = 0;
      if (!load(++ij, ir)) aborted = true;
    }
    if (aborted) break;
  }
  int cj = 0, cc = 0;
  Resolved cr;
  if (!aborted && !load(0, cr)) aborted = true;
  int* pend = nullptr;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k = 0; !aborted && cr.seg <= kSegD; ++k) {
    const int slot = k % kStages, nslot = (k + kStages - 1) % kStages;
    const bool have_next = ir.seg <= kSegD;
    bool rd = true;
    if (have_next) {
      issue_weights(ir, ic, nslot);
      rd = is_ready(ir);
    }
    cp_async_wait<kStages - 2>();
    const bool landed = mbar_wait(&bars[slot], (phase >> slot) & 1u);
    phase ^= 1u << slot;
    inflight &= ~(1u << slot);
    if (__syncthreads_or(!landed)) {
      if (tid == 0) atomicExch(status, int(MOE_ERR_TIMEOUT));
      drain();
      aborted = true;
      break;
    }
    if (tid == 0 && pend) {
      __threadfence();
      red_release_add(pend, 1);
    }
    pend = nullptr;
    const TileGeo& g = geo_of(A, cr.seg).t;
    const StageLayout L = stage_layout(g);
    uint8_t* st = smem + slot * SB;
    if (cr.U.down) {
      bool bad = false;
      if (defer & (1u << slot)) {
        defer &= ~(1u << slot);
        bad = !wait_geq(ready_ctr(A, cr.seg, cr.U.ss), Q.ngr, status);
        if (!bad) {
          const OperandSrc op = op_of(A, cr.seg);
          stage_operand_sync(g, cc, op.rowmap, cr.U.off, cr.U.cnt, op.B, op.Blo, op.Bsum, st, L);
        }
      }
      if (__syncthreads_or(bad)) {
        aborted = true;
        break;
      }
    }
    if (cc == 0) acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    compute_any<F16A>(g, cr.U.down, st, L, cr.U.cnt, acc);
    if (cc == cr.nch - 1) {
      if (cr.U.down) {
        const Sink sk = cr.seg == kSegC ? Sink{A.ysh, nullptr, H} : Sink{A.y, A.perm, H};
        write_down(sk, cr.U, acc);
        pend = ctrl + kCtlRb + cr.U.blk;
      } else {
        const bool sh = cr.seg == kSegA;
        swiglu_epilogue(acc, Ep, cr.U, I, sh ? A.sh_hh : A.hh, sh ? A.sh_hl : A.hl,
                        sh ? A.sh_hsum : A.hsum, nullptr);
        pend = ready_ctr(A, cr.seg, cr.U.ss);
      }
    }
    if (have_next) issue_operand(ir, ic, nslot, rd, defer);
    cp_async_commit();
    __syncthreads();
    if (have_next && ++ic >= ir.nch) {
      ic = 0;
      if (!load(++ij, ir)) {
        aborted = true;
        break;
      }
    }
    if (++cc >= cr.nch) {
      cc = 0;
      if (!load(++cj, cr)) {
        aborted = true;
        break;
      }
    }
  }
  if (aborted) drain();
  cp_async_wait<0>();
  if (aborted) return;
  if (tid == 0 && pend) {
    __threadfence();
    red_release_add(pend, 1);
  }

  // ---- phase 2: combine blocks
  const CombineArgs C{A.y, A.w, A.has_shared ? A.ysh : nullptr, A.has_shared ? A.sgw : nullptr,
                      A.out, 1, T, A.k, H, A.f16};
  while (cr.seg == kSegE) {
    if (tid == 0) S.flag = wait_geq(ctrl + kCtlRb + cr.U.blk, Q.nss + Q.nss_sh, status);
    __syncthreads();
    if (!S.flag) return;
    combine_block(C, cr.U.blk, 0, T);
    __syncthreads();
    if (!load(++cj, cr)) return;
  }

  // ---- exit: the last CTA zeroes the counters for the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int v = atomicAdd(ctrl + kCtlExit, 1);
    S.flag = ((v + 1) % G) == 0;
    if (S.flag) __threadfence();
  }
  __syncthreads();
  if (S.flag) {
    if (tid < 3) ctrl[kCtlRouterDone + tid] = 0;
    for (int i = kCtlReady + tid; i < kCtlEnd; i += kUnitThreads) ctrl[i] = 0;
  }
}

int stage_bytes_max(const DecodeArgs& A) {
  int sb = stage_layout(A.g13.t).bytes;
  sb = sb > stage_layout(A.g2.t).bytes ? sb : stage_layout(A.g2.t).bytes;
  if (A.has_shared) {
    sb = sb > stage_layout(A.g13s.t).bytes ? sb : stage_layout(A.g13s.t).bytes;
    sb = sb > stage_layout(A.g2s.t).bytes ? sb : stage_layout(A.g2s.t).bytes;
  }
  const int bucket = int((sizeof(SmallRouteSmem) + kStages - 1) / kStages);
  sb = sb > bucket ? sb : bucket;
  return (sb + 127) & ~127;
}

template <bool F16A>
cudaError_t launch_decode_t(const DecodeArgs& A, int sms, cudaStream_t st) {
  const int SB = stage_bytes_max(A);
  const int smem = kStages * SB;
  if (smem > kUnitSmemMax) return cudaErrorInvalidValue;
  // dynamic shared memory above 48 KiB needs an opt-in per device; raise it
  // only when a launch needs more than any earlier one on that device
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] < smem) {
    e = cudaFuncSetAttribute(k_decode<F16A>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode<F16A>, kUnitThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kUnitThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_decode<F16A>, A, SB);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int decode_smem_bytes(const DecodeArgs& A) { return kStages * stage_bytes_max(A); }

cudaError_t launch_decode(const DecodeArgs& A, int sms, cudaStream_t st) {
  return A.f16 ? launch_decode_t<true>(A, sms, st) : launch_decode_t<false>(A, sms, st);
}

}  // namespace moe
