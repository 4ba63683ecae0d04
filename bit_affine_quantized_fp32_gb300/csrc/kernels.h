// kernels.h -- internal launchers of the MoE kernels (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// One grouped-GEMV launch: for every slot (expert, bucket range) and every
// 16-row tile and k-chunk of that expert's matrix, out = W * B over the
// slot's operand rows.
struct GemvJob {
  const uint8_t* w;          // packed codes of expert 0
  const uint16_t* s;         // fp16 scales of expert 0
  const uint16_t* b;         // fp16 biases of expert 0 (nullptr for W4A16)
  long long w_estride;       // bytes of codes per expert
  long long sb_estride;      // scale entries per expert
  int rows;                  // matrix rows (multiple of 16)
  int K;                     // reduction length
  int CK;                    // k-chunk per unit (multiple of 128, divides K)
  int fmt;                   // MOE_FMT_AFFINE4_G64 / AFFINE3_G64 / W4A16_SYM_G128
  int row_bytes;             // packed bytes per matrix row
  int sb_cols;               // scale entries per matrix row (K / group)
  int sb_gran;               // cp.async granule for scale rows (4, 8 or 16 bytes)
  const int* n_slots;        // device slot count (nullptr: one fixed slot)
  const int* slot_expert;
  const int* slot_off;
  const int* slot_cnt;
  int fixed_expert;
  int fixed_cnt;
  const int* b_row;          // bucket position -> operand row (nullptr: identity)
  const uint16_t* B;         // operand rows [*, K], k-permuted bf16/fp16 bits
  const uint16_t* Blo;       // low parts for split operands (nullptr otherwise)
  const float* Bsum;         // per-64-group operand sums [*, K/64]
  float* out;                // out[(c * P + o) * rows + row]
  const int* out_idx;        // bucket position -> output row o (nullptr: identity)
  int P;                     // output rows per k-chunk plane
  int max_units;             // host upper bound on units (grid sizing)
};

int gemv_a_pitch(int fmt, int CK);
int gemv_stage_bytes(int fmt, int CK);
int gemv_smem_bytes(int fmt, int CK);

cudaError_t launch_gemv(const GemvJob& J, bool f16a, bool split, int sms, cudaStream_t st);
cudaError_t launch_hprep(const float* part, int nch, int P, int I, uint16_t* hh, uint16_t* hl,
                         float* hsum, float* hout, cudaStream_t st);
cudaError_t launch_xprep(const uint16_t* x, int T, int H, bool f16, uint16_t* xperm, float* xsum,
                         cudaStream_t st);
cudaError_t launch_combine(const float* y, const float* w, int k, const float* ysh,
                           const float* sg, int T, int H, bool f16, uint16_t* out,
                           cudaStream_t st);

// routing
struct RouterJob {
  int fmt;                   // router format: F32, BF16, AFFINE8_G64
  const void* q;
  const uint16_t* s;
  const uint16_t* b;
  int gfmt;                  // shared-gate format (gq == nullptr: none)
  const void* gq;
  const uint16_t* gs;
  const uint16_t* gb;
  const float* bias;         // [E] or nullptr
  const uint16_t* x;
  int f16;
  int T, E, H;
  float* logits;             // [T][E]
  float* gate_logit;         // [T] (when gq)
};
cudaError_t launch_router(const RouterJob& J, cudaStream_t st);
cudaError_t launch_topk(const float* logits, const float* gate_logit, int T, int E, int k,
                        int32_t* idx, float* w, float* sg, cudaStream_t st);
cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* offsets,
                          int32_t* perm, cudaStream_t st);
cudaError_t launch_slots(const int32_t* offsets, const int32_t* perm, int T, int k, int E,
                         int* nslots, int* slot_e, int* slot_off, int* slot_cnt, int* blist,
                         cudaStream_t st);

// formats
cudaError_t launch_pack(int fmt, const uint8_t* codes, int rows, int cols, uint32_t* packed,
                        cudaStream_t st);
cudaError_t launch_unpack(int fmt, const uint32_t* packed, int rows, int cols, uint8_t* codes,
                          cudaStream_t st);
cudaError_t launch_dequant(int fmt, const void* q, const uint16_t* s, const uint16_t* b, int rows,
                           int cols, float* w, cudaStream_t st);

}  // namespace moe
