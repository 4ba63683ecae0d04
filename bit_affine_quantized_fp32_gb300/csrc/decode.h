// decode.h -- arguments of the fused decode-layer kernel.
#pragma once

#include "kernels.h"

namespace moe {

// Control words (int32 indices into the workspace's control region).  They
// start at zero (moe_workspace_init); the last CTA of every fused call zeroes
// them again, except the exit counter, which only ever grows.
constexpr int kCtlXsum = 32;         // activation-sum tasks finished
constexpr int kCtlQueue = 33;        // the grid's unit queue: next entry to claim
constexpr int kCtlGen = 34;          // generation number of the last completed call
constexpr int kCtlExit = 35;         // CTAs finished (monotonic)
static_assert(kCtlWaitLimit > kCtlExit && kCtlWaitLimit < 64, "control word clash");
constexpr int kCtlReady = 64;        // [296]: 64-row h groups done per routed sub-slot
constexpr int kSharedReady = kCtlReady + 296;  // [24]: same for the shared sub-slots
constexpr int kCtlRb = kCtlReady + 320;        // [64]: down units done per 128-row block
constexpr int kCtlEnd = kCtlRb + 64;
static_assert(kCtlEnd * 4 <= kCtlTaggedOffset, "control words overlap the tagged logits");

struct DecodeArgs {
  RouterJob R;          // router, shared gate, bias, x, T, E, H, f16
  EngineCfg C;          // geo/targets: 0 routed w13, 1 routed w2, 2 shared w13, 3 shared w2
  MatSource src[4];     // operands of the four matrix slots
  int k, has_shared, KS;
  int32_t* user_idx;    // nullable outputs [T][k]
  float* user_w;
  uint16_t* out;        // [T][H]
  int* ctrl;
};

// Dynamic shared memory of a launch (S < 2: the shape does not fit).
EnginePlan decode_plan(const DecodeArgs& A);
cudaError_t launch_decode(const DecodeArgs& A, int fmt, int fmt_sh, int sms, cudaStream_t st);

}  // namespace moe
