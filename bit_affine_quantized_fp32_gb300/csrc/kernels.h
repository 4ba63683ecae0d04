// kernels.h -- internal job descriptions and launchers of the MoE kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "units.cuh"

namespace moe {

constexpr int kUnitSmemMax = 220 * 1024;

// A launch of units of one matrix family over sub-slots.
struct UnitJob {
  MatGeo g;
  int down;                 // 0: gate/up units (SwiGLU epilogue), 1: down units
  int inter;                // I
  SubSlots ss;
  OperandSrc op;
  Sink sink;                // down units: y rows
  uint16_t* hh;             // gate/up units: h outputs (k-permuted bf16 hi / lo)
  uint16_t* hl;
  float* hsum;
  float* hout;              // nullable fp32 h [rows][I]
  int max_units;            // host upper bound (grid sizing)
  int* status;              // workspace status word (bounded-wait timeouts)
};

cudaError_t launch_units(const UnitJob& J, bool f16a, int sms, cudaStream_t st);
cudaError_t launch_xprep(const uint16_t* x, int T, int H, bool f16, uint16_t* xperm, float* xsum,
                         cudaStream_t st);
cudaError_t launch_combine(const CombineArgs& A, cudaStream_t st);

// routing
struct RouterJob {
  int fmt;                  // router format: F32, BF16, F16, AFFINE8_G64
  const void* q;
  const uint16_t* s;
  const uint16_t* b;
  int gfmt;                 // shared-gate format (gq == nullptr: none)
  const void* gq;
  const uint16_t* gs;
  const uint16_t* gb;
  const float* bias;        // [E] or nullptr
  const uint16_t* x;
  int f16;
  int T, E, H;
  float* logits;            // [T][E]
  float* gate_logit;        // [T] (when gq)
};
int router_ks(int H);
int router_blocks(int E, bool gate, int H);
cudaError_t launch_router(const RouterJob& J, cudaStream_t st);
cudaError_t launch_topk(const float* logits, const float* gate_logit, int T, int E, int k,
                        int32_t* idx, float* w, float* sg, cudaStream_t st);
cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* offsets,
                          int32_t* perm, cudaStream_t st);
cudaError_t launch_subslots(const int32_t* offsets, const int32_t* perm, int T, int k, int E,
                            int* nss, int* se, int* so, int* sc, int* blist, cudaStream_t st);

// formats
cudaError_t launch_pack(int fmt, const uint8_t* codes, int rows, int cols, uint32_t* packed,
                        cudaStream_t st);
cudaError_t launch_unpack(int fmt, const uint32_t* packed, int rows, int cols, uint8_t* codes,
                          cudaStream_t st);
cudaError_t launch_dequant(int fmt, const void* q, const uint16_t* s, const uint16_t* b, int rows,
                           int cols, float* w, cudaStream_t st);
// canonical words/scales/biases of E experts <-> one tiled buffer (b unused for W4A16)
cudaError_t launch_repack(const TileGeo& g, int E, const uint32_t* wc, const uint16_t* s,
                          const uint16_t* b, uint8_t* tiled, cudaStream_t st);
cudaError_t launch_unrepack(const TileGeo& g, int E, const uint8_t* tiled, uint32_t* wc,
                            uint16_t* s, uint16_t* b, cudaStream_t st);

}  // namespace moe
