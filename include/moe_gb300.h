/*
 * moe_gb300.h -- C ABI of the routed-expert MoE layer over low-bit
 * affine-quantised weights (hand-written sm_103a CUDA kernels).
 *
 * The layer (qwen3_5 MoE 35B-A3B family: hidden 2048, 256 experts, top-8,
 * expert intermediate 512) is defined by these passages, cited by page title
 * and section:
 *   [803-gate]  "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803",
 *               comment "Progress on the 4-bit gate", paragraph "What is in it":
 *               fp32 logits over the experts and the shared-expert gate row;
 *               top-k by logit with ties to the lower id; weights exp(l - l_top)
 *               over the k; the shared expert as one more slot weighted by
 *               sigmoid(gate); the slots' fma sum rounded once; experts with a
 *               SwiGLU epilogue.
 *   [803-run]   same issue, Description, "What I want to run": MLX affine
 *               quantisation in groups of 64 -- routed experts 3-bit, the rest
 *               4-bit, router and shared-expert gate 8-bit.
 *   [w4a16]     "Sage-1.5-W4A16" model card, "Model details" / "Recipe":
 *               int4 symmetric weights, group 128, no zero point, fp16 compute.
 *   [1329]      "Sage-A1.5 (qwen3_5 MoE 35B-A3B) on the XPU backend ... #1329",
 *               Proposal: 256 experts with top-8, grouped MoE decode.
 *   [803-fp64]  same issue, "Affine experts at other widths": the loader reads
 *               MLX affine experts at further widths, checked per projection
 *               against fp64.
 *   [803-widen] same issue, comment "The 3-bit width is up as #972": the same
 *               codes at a wider width give the same results (the control).
 *   [547-win]   "Native server: --backend xpu for Nemotron on Intel Arc",
 *               update comment: a one-row window equals the decode step bit
 *               for bit; 512-row prefill windows.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller (for example
 *     allocated through PyTorch).  The library never allocates device memory.
 *   - Every call is asynchronous on the caller's cudaStream_t (0 = legacy
 *     default stream) and returns a moe_status.  Arguments are validated on
 *     the host before any launch; on an error nothing is launched and
 *     moe_last_error() names the offending argument or format.
 *   - Matrices are row-major [rows, cols] = [out, in]; quantisation groups run
 *     along cols (the reduction dimension).
 *   - Activations are bf16 or fp16 ([T, hidden]); internal arithmetic is fp32.
 *   - Pointers must be 16-byte aligned.
 *   - Scratch lives in a caller-provided workspace (moe_workspace_bytes);
 *     initialise it once with moe_workspace_init.  Calls that share a
 *     workspace must be ordered on one stream.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, bad shape, k > E, ... */
  MOE_ERR_UNSUPPORTED_FORMAT = 2,  /* a width/format this library does not read */
  MOE_ERR_WORKSPACE = 3,           /* workspace missing or too small */
  MOE_ERR_CUDA = 4,                /* a CUDA runtime call failed */
  MOE_ERR_TIMEOUT = 5,             /* a bounded device-side wait gave up */
  MOE_ERR_MISALIGNED = 6,          /* a pointer is not 16-byte aligned */
  MOE_ERR_RANGE = 7                /* device status: an activation or h value of the prefill
                                      form lay outside fp16's range (its operands are fp16) */
} moe_status;

/* Storage formats.  Quantised formats hold packed codes in little-endian
 * uint32 words plus fp16 scales [rows, cols/G] (and fp16 biases for affine):
 *   AFFINE8_G64  MLX affine 8-bit, 4 codes per word, code i at bits [8i, 8i+8)
 *   AFFINE4_G64  MLX affine 4-bit, 8 codes per word, code i at bits [4i, 4i+4)
 *   AFFINE3_G64  MLX affine 3-bit: each row is one LSB-first bit stream, code
 *                c at stream bits [3c, 3c+3) (codes may straddle two words;
 *                32 codes fill 3 words exactly)
 *   AFFINE2_G64, AFFINE5_G64, AFFINE6_G64  MLX affine at the other widths the
 *                pages' loader reads, rows as LSB-first bit streams as for
 *                3-bit (code c at bits [bc, bc+b)); 2-bit is 16 codes per word
 *     affine dequantisation: w = scale * q + bias, q unsigned   [803-run],
 *                                                                [803-fp64]
 *   W4A16_SYM_G128  compressed-tensors pack-quantized int4: 8 nibbles per
 *                word LSB-first, stored u = q + 8 (q in -8..7), w = scale * q,
 *                no bias                                          [w4a16]
 */
typedef enum moe_format {
  MOE_FMT_F32 = 0,
  MOE_FMT_BF16 = 1,
  MOE_FMT_F16 = 2,
  MOE_FMT_AFFINE8_G64 = 3,
  MOE_FMT_AFFINE4_G64 = 4,
  MOE_FMT_AFFINE3_G64 = 5,
  MOE_FMT_W4A16_SYM_G128 = 6,
  MOE_FMT_AFFINE2_G64 = 7,
  MOE_FMT_AFFINE5_G64 = 8,
  MOE_FMT_AFFINE6_G64 = 9
} moe_format;

/* One matrix [rows, cols] in any format.  For F32/BF16/F16 qweight holds the
 * values and scales/biases are NULL; biases is NULL for W4A16. */
typedef struct moe_qmatrix {
  int32_t fmt;
  int32_t rows;
  int32_t cols;
  int32_t reserved;
  const void* qweight;
  const void* scales;
  const void* biases;
} moe_qmatrix;

/* Storage layouts of an expert bank. */
typedef enum moe_layout {
  MOE_LAYOUT_CANONICAL = 0, /* the format's own row-major words + scale tables */
  MOE_LAYOUT_TILED = 1      /* kernel-tiled (moe_repack_bank), read by the expert kernels */
} moe_layout;

/* n_experts experts in one quantised format.
 * CANONICAL layout, stacked contiguously:
 *   w13 [E][2*inter][hidden] : gate rows 0..inter-1, then up rows
 *   w2  [E][hidden][inter]   : down projection
 * with s13/b13 and s2/b2 their fp16 scales/biases ([E][rows][cols/G]).
 * TILED layout (produced by moe_repack_bank): w13 and w2 each point at one
 * buffer of moe_tiled_bytes() bytes holding codes, scales and biases cut
 * into per-(expert, 128-row block, k-chunk) blocks in MMA fragment order;
 * s13/b13/s2/b2 are NULL.  The expert kernels read TILED banks only.  */
typedef struct moe_expert_bank {
  int32_t fmt;
  int32_t n_experts;
  int32_t inter;
  int32_t hidden;
  int32_t layout;   /* moe_layout */
  int32_t reserved;
  const void* w13;
  const void* s13;
  const void* b13;
  const void* w2;
  const void* s2;
  const void* b2;
} moe_expert_bank;

/* flags of moe_experts_forward / moe_layer_forward */
#define MOE_FLAG_FORCE_DECODE 1   /* use the decode (grouped GEMV) form at any T */
#define MOE_FLAG_UNFUSED 2        /* moe_layer_forward: one launch per step instead of the
                                     single persistent decode launch (same results) */
#define MOE_FLAG_FORCE_PREFILL 8  /* use the prefill form (tcgen05 expert GEMMs) at any
                                     T >= 1; experts in AFFINE3/4_G64 or W4A16 only
                                     (others: MOE_ERR_UNSUPPORTED_FORMAT); not together
                                     with MOE_FLAG_FORCE_DECODE */
/* The engine's bf16 rounding chain ([803-gate]: router and combine checked
 * byte-equal against a host reference, weights within a bf16 step).  In
 * moe_route and moe_layer_forward: the router and shared-gate rows are
 * rounded to bf16 (through their fp32 value, nearest, ties to even) before
 * the dot products, each slot weight is stored as bf16(w), and the shared
 * weight as bf16(sigmoid(bf16(g))); logits, softmax and sums stay fp32.  In
 * moe_experts_forward (and the layer's combine): the given slot and shared
 * weights are rounded to bf16 before the fp32 fma chain (a no-op on weights
 * moe_route already rounded).  Without the flag the weights stay fp32 and
 * the only rounding is the final cast to the activation type.            */
#define MOE_FLAG_ROUND_BF16 4

/* The decode form (grouped GEMV on exact integer codes) serves n_tokens <=
 * MOE_DECODE_MAX_TOKENS; above it the prefill form runs the expert GEMMs on
 * the tensor cores (tcgen05) over tiles of up to 128 tokens of one expert,
 * with fp16 operands -- the dequantised weights fma(s, q, b) rounded once,
 * the activations converted to fp16 (exact within fp16's normal range), h
 * stored as fp16 -- and fp32 accumulation: the same values to within the
 * layer's tolerance, not the same bits as the decode form.  Experts with at
 * most 16 assignments in the call run the decode form's units, on a second
 * stream (one per CUDA context and caller stream, created on first use)
 * that forks from the caller's stream with an event and joins it again
 * before the combine, so the call stays capturable in a CUDA graph. */
#define MOE_DECODE_MAX_TOKENS 32

/* Human-readable name of a status; never NULL. */
const char* moe_status_string(moe_status s);

/* Detail of the last error returned on this host thread ("" if none). */
const char* moe_last_error(void);

/* Bytes of workspace needed for calls with up to max_tokens tokens and the
 * given shape.  Returns 0 on invalid arguments. */
size_t moe_workspace_bytes(int max_tokens, int n_experts, int top_k, int hidden, int inter);

/* Zero the workspace's control words (status, counters).  Call once after
 * allocating a workspace, before its first use, and again after a call
 * reported MOE_ERR_TIMEOUT through moe_get_device_status. */
moe_status moe_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/* Limit of every bounded device-side wait (a CTA waiting for another CTA's
 * results, or for its own copies) of later calls on this workspace, in
 * microseconds; 0 restores the default of one second.  A wait that runs out
 * records MOE_ERR_TIMEOUT in the workspace's status word and makes the rest
 * of its CTA's waits return at once, so the launch ends (its outputs are then
 * garbage); the workspace must be re-initialised before the next call.  The
 * pages' counterpart is the serving engine's wall-clock guard with an error
 * event on shutdown ([547-win]).  Stream-ordered (a one-thread kernel writes
 * the control word); moe_workspace_init resets it to the default.
 *   limit_us  0 .. 2^31 - 1, else MOE_ERR_INVALID_ARG.                   */
moe_status moe_workspace_set_wait_limit(void* ws, size_t ws_bytes, unsigned limit_us,
                                        cudaStream_t stream);

/* Read and clear the device status word of a workspace (synchronises the
 * stream).  *device_status receives MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_RANGE
 * (the prefill form met an activation or h value beyond fp16's range; its
 * outputs are then not valid -- the decode form, MOE_FLAG_FORCE_DECODE, has
 * no such limit). */
moe_status moe_get_device_status(void* ws, size_t ws_bytes, int* device_status,
                                 cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Routing [803-gate], [1329].
 *
 * moe_route computes, for each token t of x [T, hidden]:
 *   l[t, e] = sum_h W_r[e, h] * x[t, h] + logit_bias[e]      (fp32)
 *   slots 0..k-1 = the k experts ordered by (logit desc, id asc); NaN ranks
 *                  below every number, NaNs among themselves by id
 *   w[t, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0)          (fp32)
 *   shared_gate_w[t] = 1 / (1 + exp(-sum_h g[h] x[t, h]))    (if shared_gate)
 * and buckets the assignments a = t*k + j by expert: bucket_offsets [E+1]
 * (exclusive prefix sum of the per-expert counts) and bucket_perm [T*k] (the
 * assignment ids sorted by expert, ascending a within an expert).
 *   router       [E, hidden] in F32, BF16 or AFFINE8_G64
 *   logit_bias   nullable [E] fp32 per-expert logit offset
 *   shared_gate  nullable [1, hidden] in F32, BF16 or AFFINE8_G64
 *   act          MOE_FMT_BF16 or MOE_FMT_F16 (type of x)
 *   top_k        1..8, <= E;  E <= 256
 *   logits       nullable [T, E] fp32 output
 *   topk_idx [T, k] int32, topk_w [T, k] fp32, shared_gate_w nullable [T]
 *   flags        0 or MOE_FLAG_ROUND_BF16 (the engine's bf16 rounding chain)
 * Above MOE_DECODE_MAX_TOKENS the logits come from the tensor cores: each
 * router (and gate) weight split exactly into three bf16 parts, fp16
 * activations into two, so every product is exact and the sums are fp32
 * (four k-slices added in order); below it a SIMT fp32 dot product.  Both
 * lie within the fp32 dot-product bound of the exact logits.
 */
moe_status moe_route(const moe_qmatrix* router, const float* logit_bias,
                     const moe_qmatrix* shared_gate, const void* x, int act, int n_tokens,
                     int top_k, float* logits, int32_t* topk_idx, float* topk_w,
                     float* shared_gate_w, int32_t* bucket_offsets, int32_t* bucket_perm,
                     int flags, void* ws, size_t ws_bytes, cudaStream_t stream);

/* moe_route without a workspace, for callers that cannot hand the library
 * memory (no device allocator of their own, or no allocation allowed once
 * serving).  The pages have no counterpart to this entry point: it is
 * moe_route (same kernels, same results) with its one scratch buffer -- the
 * fp32 logits between the router and top-k kernels -- in a static device
 * array of 32 * 256 + 32 floats; no logits output.  The array belongs to the
 * library's module as loaded into a CUDA context, so there is one copy per
 * context (module instance), not per device.
 *   Limits: n_tokens <= 32 and n_tokens * experts <= 8192, else
 *           MOE_ERR_WORKSPACE before anything is launched.
 *   The first call in a context looks the array's address up (a synchronous
 *   runtime query, cached under the context's id; after cudaDeviceReset or in
 *   another context it is looked up again), so make it before any stream
 *   capture.
 *   Nothing in the array needs to start at zero.  Calls that overlap in time
 *   within one context (other streams, other host threads) race on it. */
moe_status moe_route_static(const moe_qmatrix* router, const float* logit_bias,
                            const moe_qmatrix* shared_gate, const void* x, int act,
                            int n_tokens, int top_k, int32_t* topk_idx, float* topk_w,
                            float* shared_gate_w, int32_t* bucket_offsets, int32_t* bucket_perm,
                            cudaStream_t stream);

/* Top-k + weights from given fp32 logits [T, E] (same rules as moe_route). */
moe_status moe_topk_softmax(const float* logits, int n_tokens, int n_experts, int top_k,
                            int32_t* topk_idx, float* topk_w, cudaStream_t stream);

/* Bucketing alone: counting sort of topk_idx [T, k] by expert (see moe_route). */
moe_status moe_bucket(const int32_t* topk_idx, int n_tokens, int top_k, int n_experts,
                      int32_t* bucket_offsets, int32_t* bucket_perm, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Experts [803-gate]: for an expert with gate Wg, up Wu (rows of w13) and down
 * Wd (w2):  h = silu(Wg x) * (Wu x),  y = Wd h  (fp32 accumulation).
 *
 * moe_expert_mlp runs expert `expert` of `bank` on all n_tokens rows of x:
 *   h_out nullable [T, inter] fp32, y_out [T, hidden] fp32.
 * moe_shared_expert is the same for expert 0 of a one-expert bank:
 *   y_shared [T, hidden] fp32.
 * Banks must be TILED (moe_repack_bank).  Formats: AFFINE2/3/4/5/6/8_G64
 * (hidden and inter multiples of 128), W4A16_SYM_G128 (multiples of 256);
 * inter <= 512.  Every width computes sum_i q_i x_i on the exact integer
 * codes with one fp32 accumulation order, so the same codes stored at any
 * affine width give bit-identical results ([803-widen]).  The fused decode
 * launch and the prefill tensor-core GEMMs read AFFINE3/4_G64 and W4A16; the
 * other widths run the launch-per-step decode form at any n_tokens (the same
 * results the fused launch would give).
 */
moe_status moe_expert_mlp(const moe_expert_bank* bank, int expert, const void* x, int act,
                          int n_tokens, float* h_out, float* y_out, void* ws, size_t ws_bytes,
                          cudaStream_t stream);

moe_status moe_shared_expert(const moe_expert_bank* shared, const void* x, int act,
                             int n_tokens, float* y_shared, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* The routed experts and the combine [803-gate]:
 *   out[t, :] = round( sum_{j<k} w[t, j] * y_{t,j} + s_t * y_shared[t, :] )
 * an fp32 fma chain in slot order with the shared slot last, rounded once to
 * the activation type.  y_shared/shared_gate_w nullable (no shared slot when
 * y_shared is NULL; weight 1 when only shared_gate_w is NULL).
 * Routing inputs are moe_route's outputs (or any valid equivalent).
 * flags: MOE_FLAG_FORCE_DECODE, MOE_FLAG_FORCE_PREFILL, MOE_FLAG_ROUND_BF16
 * (weights rounded to bf16 before the sum).
 * In the decode form every token's output row depends only on that token's
 * inputs: a row is bit-identical whatever the other rows of the call
 * ([547-win]); the prefill form (T > 32) matches it to within the layer's
 * tolerance.                                                             */
moe_status moe_experts_forward(const moe_expert_bank* experts, const void* x, int act,
                               int n_tokens, int top_k, const int32_t* topk_idx,
                               const float* topk_w, const int32_t* bucket_offsets,
                               const int32_t* bucket_perm, const float* y_shared,
                               const float* shared_gate_w, void* out, int flags, void* ws,
                               size_t ws_bytes, cudaStream_t stream);

/* The whole layer in one call: route, shared expert, routed experts, combine.
 * shared (nullable) is a one-expert bank; shared_gate nullable.
 * topk_idx/topk_w nullable outputs [T, k].
 * flags: MOE_FLAG_FORCE_DECODE, MOE_FLAG_FORCE_PREFILL, MOE_FLAG_UNFUSED,
 * MOE_FLAG_ROUND_BF16.
 * For n_tokens <= MOE_DECODE_MAX_TOKENS the layer runs as ONE persistent
 * cooperative launch (one CTA per SM) whose phases synchronise through
 * counters in the workspace; every wait is bounded and reports
 * MOE_ERR_TIMEOUT in the workspace status word instead of hanging.  The
 * results are bit-identical to the multi-launch path (MOE_FLAG_UNFUSED).
 * Above it, a shared expert of the routed experts' format runs inside the
 * routed experts' two tensor-core GEMM launches (its units first). */
moe_status moe_layer_forward(const moe_qmatrix* router, const float* logit_bias,
                             const moe_qmatrix* shared_gate, const moe_expert_bank* experts,
                             const moe_expert_bank* shared, const void* x, int act,
                             int n_tokens, int top_k, void* out, int32_t* topk_idx,
                             float* topk_w, int flags, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Pack / unpack / dequantise, one pair per quantised format [803-run],
 * [w4a16].  codes are [rows, cols] bytes: unsigned 0..2^bits-1 for affine,
 * signed -8..7 (int8) for W4A16.  packed is [rows, cols*bits/32] uint32.
 * cols must be a multiple of 32.  A code out of range sets the packed word
 * to the low bits of the code (no error is reported on the device).     */
moe_status moe_pack_affine8_g64(const uint8_t* codes, int rows, int cols, uint32_t* packed,
                                cudaStream_t stream);
moe_status moe_unpack_affine8_g64(const uint32_t* packed, int rows, int cols, uint8_t* codes,
                                  cudaStream_t stream);
moe_status moe_pack_affine4_g64(const uint8_t* codes, int rows, int cols, uint32_t* packed,
                                cudaStream_t stream);
moe_status moe_unpack_affine4_g64(const uint32_t* packed, int rows, int cols, uint8_t* codes,
                                  cudaStream_t stream);
moe_status moe_pack_affine3_g64(const uint8_t* codes, int rows, int cols, uint32_t* packed,
                                cudaStream_t stream);
moe_status moe_unpack_affine3_g64(const uint32_t* packed, int rows, int cols, uint8_t* codes,
                                  cudaStream_t stream);
moe_status moe_pack_w4a16_g128(const int8_t* codes, int rows, int cols, uint32_t* packed,
                               cudaStream_t stream);
moe_status moe_unpack_w4a16_g128(const uint32_t* packed, int rows, int cols, int8_t* codes,
                                 cudaStream_t stream);
/* The other MLX affine widths ([803-fp64]): codes 0 .. 2^bits - 1. */
moe_status moe_pack_affine2_g64(const uint8_t* codes, int rows, int cols, uint32_t* packed,
                                cudaStream_t stream);
moe_status moe_unpack_affine2_g64(const uint32_t* packed, int rows, int cols, uint8_t* codes,
                                  cudaStream_t stream);
moe_status moe_pack_affine5_g64(const uint8_t* codes, int rows, int cols, uint32_t* packed,
                                cudaStream_t stream);
moe_status moe_unpack_affine5_g64(const uint32_t* packed, int rows, int cols, uint8_t* codes,
                                  cudaStream_t stream);
moe_status moe_pack_affine6_g64(const uint8_t* codes, int rows, int cols, uint32_t* packed,
                                cudaStream_t stream);
moe_status moe_unpack_affine6_g64(const uint32_t* packed, int rows, int cols, uint8_t* codes,
                                  cudaStream_t stream);

/* Kernel-tiled expert layout.  The pages' engine likewise keeps its experts
 * in kernel tables of its own (gate and up interleaved per group, "Progress
 * on the 4-bit gate" comment of "qwen3_5_moe on native CUDA with 3-bit routed
 * experts ... #803").  A TILED bank holds exactly the canonical bank's codes,
 * scales and biases, rearranged (the 3-bit codes as bit planes, 3 bits each).
 *   moe_tiled_bytes    bytes of the w13 (which = 0) or w2 (which = 1) buffer
 *                      of a TILED bank; 0 on invalid arguments.
 *   moe_repack_bank    CANONICAL bank -> the two TILED buffers (device).
 *   moe_unrepack_bank  TILED bank -> canonical words/scales/biases
 *                      (b13/b2 ignored for W4A16); unrepack(repack(x)) == x. */
size_t moe_tiled_bytes(int fmt, int n_experts, int inter, int hidden, int which);
moe_status moe_repack_bank(const moe_expert_bank* canonical, void* w13_tiled, void* w2_tiled,
                           cudaStream_t stream);
moe_status moe_unrepack_bank(const moe_expert_bank* tiled, void* w13, void* s13, void* b13,
                             void* w2, void* s2, void* b2, cudaStream_t stream);

/* Dequantise any matrix to fp32: w = fmaf(scale, q, bias) for affine (the
 * exact value scale*q + bias rounded once to fp32) or scale * q for W4A16
 * (exact); F32/BF16/F16 values are widened.  w is [rows, cols] fp32.    */
moe_status moe_dequant(const moe_qmatrix* m, float* w, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
