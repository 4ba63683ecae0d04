// decode.h -- arguments of the fused decode-layer kernel.
#pragma once

#include "kernels.h"

namespace moe {

// Control words (int32 indices into the workspace's control region).  They
// start at zero (moe_workspace_init); the last CTA of every fused call zeroes
// them again, except the exit counter, which only ever grows.
constexpr int kCtlStatus = 0;
constexpr int kCtlRouterDone = 32;    // router blocks finished
constexpr int kCtlXprepDone = 33;     // x-preparation blocks finished
constexpr int kCtlRoutingReady = 34;  // 1 once routing and sub-slots are written
constexpr int kCtlExit = 35;          // CTAs finished (monotonic)
constexpr int kMaxSubFused = 296;     // routed sub-slots of a fused call (T <= 32)
constexpr int kCtlReady = 64;         // [320]: 64-row h groups done per sub-slot
constexpr int kSharedReady = kCtlReady + kMaxSubFused;  // shared-expert sub-slots
constexpr int kCtlRb = kCtlReady + 320;                 // [64]: down units done per block
constexpr int kCtlEnd = kCtlRb + 64;
constexpr int kCtlBytes = 16384;
static_assert(kCtlEnd * 4 <= kCtlBytes, "control region too small");

struct DecodeArgs {
  RouterJob R;                 // router, shared gate, x, T, E, H, logits, gate logits
  int k, inter, f16, has_shared;
  int KS, NR, XB;              // router k-splits, router blocks, x-prep blocks
  MatGeo g13, g2, g13s, g2s;   // routed and shared matrices
  uint16_t* xperm;
  float* xsum;
  int32_t* idx;
  float* w;
  float* sgw;                  // nullptr without a shared gate
  int32_t* offsets;
  int32_t* perm;
  int* nss;
  int* se;
  int* so;
  int* sc;
  int* rows;                   // [sub-slot][8] token ids
  int* blist;
  uint16_t* hh;
  uint16_t* hl;
  float* hsum;
  float* y;
  uint16_t* sh_hh;
  uint16_t* sh_hl;
  float* sh_hsum;
  float* ysh;
  int32_t* user_idx;           // nullable outputs
  float* user_w;
  uint16_t* out;
  int* ctrl;
};

int decode_smem_bytes(const DecodeArgs& A);
cudaError_t launch_decode(const DecodeArgs& A, int sms, cudaStream_t st);

}  // namespace moe
