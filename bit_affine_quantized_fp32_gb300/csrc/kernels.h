// kernels.h -- internal job descriptions and launchers of the MoE kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "engine.cuh"

namespace moe {

// Sub-slot list of a standalone job: sub-slot ss holds tokens [off, off + cnt)
// of expert e, in bucket positions (a table written by k_subslots) -- or, for
// a fixed expert over T tokens, sub-slot ss is tokens [8 ss, min(T, 8 ss + 8)).
struct SubSlots {
  const int* n;  // device count (nullptr: fixed expert)
  const int* e;
  const int* off;
  const int* cnt;
  int fixed_e;
  int fixed_T;
};

// A standalone launch of units of one matrix family (slot `mat`, 0 = w13 or
// 1 = w2 of the bank in C.geo[0..1]) over a sub-slot list.
struct UnitJob {
  EngineCfg C;
  MatSource src;       // operand rows of `mat`
  int mat;
  int rows;            // kRowsDirect / kRowsGather / kRowsScatter
  SubSlots ss;
  const int* perm;     // bucket position -> assignment id (Gather / Scatter)
  int k;
  int max_units;       // host upper bound (grid sizing)
};

cudaError_t launch_units(const UnitJob& J, bool f16a, int sms, cudaStream_t st);
cudaError_t launch_xsum(const uint16_t* x, int T, int H, bool f16, const TileGeo& g13,
                        float* xsum, cudaStream_t st);
// launch_xsum over bf16 activations that also writes their fp16 copy xh
// (MOE_ERR_RANGE in *status for a value outside fp16's range)
cudaError_t launch_xsum_f16(const uint16_t* x, int T, int H, const TileGeo& g13, float* xsum,
                            uint16_t* xh, int* status, cudaStream_t st);

struct CombineArgs {
  const float* y;    // [2][T*k][H] k-half planes
  size_t yhalf;      // elements to the second plane
  const float* w;    // [T][k]
  const float* ysh;  // [T][H] or nullptr
  const float* ysh2; // second plane of ysh, or nullptr when ysh is final
  const float* sg;   // [T] or nullptr (weight 1)
  uint16_t* out;     // [T][H]
  int T, k, H, f16;
  int round_bf16;    // w and sg rounded to bf16 before the sum
  const int32_t* idx;      // prefill form (nullable): the assignments' experts [T][k]
  const int32_t* offsets;  //   and bucket offsets [E+1]; experts with more than
  int one_plane_max;       //   one_plane_max assignments have y in plane 0 only
};
cudaError_t launch_combine(const CombineArgs& A, cudaStream_t st);
// *p = v, stream-ordered (a workspace control word)
cudaError_t launch_store_word(int* p, int v, cudaStream_t st);
cudaError_t launch_add_planes(const float* a, const float* b, float* dst, long n,
                              cudaStream_t st);

// Dynamic shared memory of an engine kernel for the given matrices: two
// operand buffers when they fit (else one), then as many weight stages as fit
// (at most kMaxStages).  S < 2 means the shape does not fit.
struct EnginePlan {
  int OB, nob, SB, S;
  int bytes() const { return nob * OB + S * SB; }
};
EnginePlan engine_plan(const TileGeo* geos, int n, int static_bytes);

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
  int round_bf16;           // router and gate rows rounded to bf16 before the dot products
  float* part;              // nullable scratch [4][T][E + 1]: the tensor-core router's
                            // k-slice sums (used for T > 32)
  uint16_t* split;          // scratch with part: bf16 parts of the weights [3][E + 1][H]
                            // then of fp16 x [2][T][H]
};
// elements of RouterJob::split for T tokens, E experts (+ 1 gate row), H columns
inline size_t router_split_elems(long T, long E, long H) { return size_t(3 * (E + 1) * H + 2 * T * H); }
int router_ks(int H);
int router_blocks(int E, bool gate, int H);
// the SIMT router (logits and gate logit of every token)
cudaError_t launch_router(const RouterJob& J, cudaStream_t st);
// round_bf16: slot weights bf16(w) and shared weight bf16(sigmoid(bf16(g)))
// launch_router then launch_topk (same results); above 32 tokens the
// tensor-core router's k-slice sums feed the top-k directly (logits and gate
// logit still written).  sg is used only with a gate row.
cudaError_t launch_router_topk(const RouterJob& J, int k, int32_t* idx, float* w, float* sg,
                               bool round_bf16, cudaStream_t st);
cudaError_t launch_topk(const float* logits, const float* gate_logit, int T, int E, int k,
                        int32_t* idx, float* w, float* sg, bool round_bf16, cudaStream_t st);
cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* offsets,
                          int32_t* perm, cudaStream_t st);
// Sub-slots (runs of at most `run` bucket positions) of the experts with
// more than cmin and at most cmax assignments.
cudaError_t launch_subslots(const int32_t* offsets, int E, int* nss, int* se, int* so, int* sc,
                            cudaStream_t st, int run = kMaxTok, int cmin = 0, int cmax = 1 << 30);
// A sub-slot table in device memory: count, then expert / first position /
// rows of each entry.
struct SubslotTable {
  int* n;
  int* e;
  int* off;
  int* cnt;
};
// Table A: runs of run_a positions of the experts with more than `split`
// assignments; table B: runs of run_b of the experts with 1..split.
cudaError_t launch_subslots_pair(const int32_t* offsets, int E, int split, const SubslotTable& A,
                                 int run_a, const SubslotTable& B, int run_b, cudaStream_t st);
// launch_bucket then launch_subslots_pair, in one launch
cudaError_t launch_bucket_tables(const int32_t* idx, int T, int k, int E, int32_t* offsets,
                                 int32_t* perm, int split, const SubslotTable& A, int run_a,
                                 const SubslotTable& B, int run_b, cudaStream_t st);

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
