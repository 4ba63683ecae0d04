// capi.cu -- the extern "C" entry points: argument validation on the host,
// workspace layout, and kernel launches on the caller's stream.
//
// Unsupported widths are refused by name before anything is launched, as the
// loader of "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803"
// refuses any width its kernels do not read (comment "Progress on the 4-bit
// gate", last paragraph).

#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace moe {
int router_ks(int H);
}

using namespace moe;

namespace {

thread_local char g_err[512] = "";

moe_status fail(moe_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

moe_status ok() {
  g_err[0] = 0;
  return MOE_OK;
}

moe_status cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define MOE_CUDA(call, where)                 \
  do {                                        \
    cudaError_t e_ = (call);                  \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

const char* fmt_name(int f) {
  switch (f) {
    case MOE_FMT_F32: return "F32";
    case MOE_FMT_BF16: return "BF16";
    case MOE_FMT_F16: return "F16";
    case MOE_FMT_AFFINE8_G64: return "AFFINE8_G64";
    case MOE_FMT_AFFINE4_G64: return "AFFINE4_G64";
    case MOE_FMT_AFFINE3_G64: return "AFFINE3_G64";
    case MOE_FMT_W4A16_SYM_G128: return "W4A16_SYM_G128";
    default: return "unknown";
  }
}

int fmt_bits(int f) {
  switch (f) {
    case MOE_FMT_AFFINE8_G64: return 8;
    case MOE_FMT_AFFINE4_G64: return 4;
    case MOE_FMT_AFFINE3_G64: return 3;
    case MOE_FMT_W4A16_SYM_G128: return 4;
    default: return 0;
  }
}

int fmt_group(int f) { return f == MOE_FMT_W4A16_SYM_G128 ? 128 : 64; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

moe_status check_act(int act) {
  if (act != MOE_FMT_BF16 && act != MOE_FMT_F16)
    return fail(MOE_ERR_UNSUPPORTED_FORMAT,
                "activation format %s (%d) is not read; use BF16 or F16", fmt_name(act), act);
  return MOE_OK;
}

// Router / shared-gate matrix: F32, BF16, F16 or AFFINE8_G64.
moe_status check_router_matrix(const moe_qmatrix* m, const char* what, int rows, int H) {
  if (!m) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", what);
  if (m->fmt != MOE_FMT_F32 && m->fmt != MOE_FMT_BF16 && m->fmt != MOE_FMT_F16 &&
      m->fmt != MOE_FMT_AFFINE8_G64)
    return fail(MOE_ERR_UNSUPPORTED_FORMAT, "%s format %s (%d) is not read by the router kernel",
                what, fmt_name(m->fmt), m->fmt);
  if (rows >= 0 && m->rows != rows)
    return fail(MOE_ERR_INVALID_ARG, "%s has %d rows, expected %d", what, m->rows, rows);
  if (m->cols != H) return fail(MOE_ERR_INVALID_ARG, "%s has %d cols, expected %d", what, m->cols, H);
  if (!m->qweight) return fail(MOE_ERR_INVALID_ARG, "%s qweight is NULL", what);
  if (!aligned16(m->qweight)) return fail(MOE_ERR_MISALIGNED, "%s qweight not 16-byte aligned", what);
  if (m->fmt == MOE_FMT_AFFINE8_G64) {
    if (!m->scales || !m->biases)
      return fail(MOE_ERR_INVALID_ARG, "%s: AFFINE8_G64 needs scales and biases", what);
    if (!aligned4(m->scales) || !aligned4(m->biases))
      return fail(MOE_ERR_MISALIGNED, "%s scales/biases not 4-byte aligned", what);
  }
  return MOE_OK;
}

moe_status check_hidden(int H) {
  if (H <= 0 || H % 128 != 0 || router_ks(H) == 0)
    return fail(MOE_ERR_INVALID_ARG,
                "hidden=%d unsupported by the router kernel (a multiple of 128 that splits into "
                "at most 8 parts of at most 512)",
                H);
  return MOE_OK;
}

moe_status check_bank(const moe_expert_bank* b, const char* what) {
  if (!b) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", what);
  const int f = b->fmt;
  if (f != MOE_FMT_AFFINE4_G64 && f != MOE_FMT_AFFINE3_G64 && f != MOE_FMT_W4A16_SYM_G128)
    return fail(MOE_ERR_UNSUPPORTED_FORMAT,
                "%s: expert format %s (%d) is not read by the expert kernels (AFFINE4_G64, "
                "AFFINE3_G64, W4A16_SYM_G128 are)",
                what, fmt_name(f), f);
  if (b->n_experts <= 0 || b->n_experts > 256)
    return fail(MOE_ERR_INVALID_ARG, "%s: n_experts=%d not in 1..256", what, b->n_experts);
  const int H = b->hidden, I = b->inter;
  const int q = f == MOE_FMT_W4A16_SYM_G128 ? 256 : 128;
  if (H <= 0 || H % q != 0 || I <= 0 || I % q != 0)
    return fail(MOE_ERR_INVALID_ARG, "%s: hidden=%d and inter=%d must be multiples of %d for %s",
                what, H, I, q, fmt_name(f));
  if (I > 1024) return fail(MOE_ERR_INVALID_ARG, "%s: inter=%d > 1024 unsupported", what, I);
  if (H > 8192) return fail(MOE_ERR_INVALID_ARG, "%s: hidden=%d > 8192 unsupported", what, H);
  if (!b->w13 || !b->s13 || !b->w2 || !b->s2)
    return fail(MOE_ERR_INVALID_ARG, "%s: weight or scale pointer is NULL", what);
  if (f != MOE_FMT_W4A16_SYM_G128 && (!b->b13 || !b->b2))
    return fail(MOE_ERR_INVALID_ARG, "%s: affine format needs biases", what);
  if (!aligned16(b->w13) || !aligned16(b->w2) || !aligned16(b->s13) || !aligned16(b->s2) ||
      (b->b13 && !aligned16(b->b13)) || (b->b2 && !aligned16(b->b2)))
    return fail(MOE_ERR_MISALIGNED, "%s: weight/scale/bias pointers must be 16-byte aligned", what);
  return MOE_OK;
}

int sb_granule(int bytes_row, int bytes_chunk) {
  for (int g = 16; g >= 4; g >>= 1)
    if (bytes_row % g == 0 && bytes_chunk % g == 0) return g;
  return 0;
}

// GEMV job for gate/up (w13) or down (w2) of a bank.
GemvJob bank_job(const moe_expert_bank* b, bool down) {
  GemvJob J{};
  const int f = b->fmt, H = b->hidden, I = b->inter;
  const int G = fmt_group(f), bits = fmt_bits(f);
  J.fmt = f;
  J.rows = down ? H : 2 * I;
  J.K = down ? I : H;
  J.CK = down ? I : gu_chunk(H);
  J.row_bytes = J.K * bits / 8;
  J.sb_cols = J.K / G;
  J.sb_gran = sb_granule(J.sb_cols * 2, (J.CK / G) * 2);
  J.w = static_cast<const uint8_t*>(down ? b->w2 : b->w13);
  J.s = static_cast<const uint16_t*>(down ? b->s2 : b->s13);
  J.b = f == MOE_FMT_W4A16_SYM_G128 ? nullptr : static_cast<const uint16_t*>(down ? b->b2 : b->b13);
  J.w_estride = (long long)J.rows * J.row_bytes;
  J.sb_estride = (long long)J.rows * J.sb_cols;
  return J;
}

char* wsp(void* ws, size_t off) { return static_cast<char*>(ws) + off; }

moe_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned16(ws)) return fail(MOE_ERR_MISALIGNED, "workspace not 16-byte aligned");
  if (ws_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, this call needs %zu", ws_bytes, need);
  return MOE_OK;
}

// One expert (a fixed slot holding every token) over the T rows of x, with
// the given workspace layout: x prep -> gate/up GEMV -> SwiGLU -> down GEMV.
moe_status run_expert_mlp(const moe_expert_bank* bank, int expert, const void* x, bool f16,
                          int T, float* h_out, float* y_out, void* ws, const WsLayout& L,
                          cudaStream_t stream) {
  const int sms = sm_count();
  const int H = bank->hidden, I = bank->inter;
  MOE_CUDA(launch_xprep(static_cast<const uint16_t*>(x), T, H, f16,
                        reinterpret_cast<uint16_t*>(wsp(ws, L.xperm)),
                        reinterpret_cast<float*>(wsp(ws, L.xsum)), stream),
           "x prep");
  GemvJob J = bank_job(bank, false);
  J.fixed_expert = expert;
  J.fixed_cnt = T;
  J.B = reinterpret_cast<const uint16_t*>(wsp(ws, L.xperm));
  J.Bsum = reinterpret_cast<const float*>(wsp(ws, L.xsum));
  J.out = reinterpret_cast<float*>(wsp(ws, L.sh_part));
  J.P = T;
  J.max_units = (J.rows / 16) * (J.K / J.CK);
  MOE_CUDA(launch_gemv(J, f16, false, sms, stream), "gate/up kernel");
  const int nch = H / J.CK;
  MOE_CUDA(launch_hprep(reinterpret_cast<const float*>(wsp(ws, L.sh_part)), nch, T, I,
                        reinterpret_cast<uint16_t*>(wsp(ws, L.sh_hh)),
                        reinterpret_cast<uint16_t*>(wsp(ws, L.sh_hl)),
                        reinterpret_cast<float*>(wsp(ws, L.sh_hsum)), h_out, stream),
           "swiglu kernel");
  GemvJob D = bank_job(bank, true);
  D.fixed_expert = expert;
  D.fixed_cnt = T;
  D.B = reinterpret_cast<const uint16_t*>(wsp(ws, L.sh_hh));
  D.Blo = reinterpret_cast<const uint16_t*>(wsp(ws, L.sh_hl));
  D.Bsum = reinterpret_cast<const float*>(wsp(ws, L.sh_hsum));
  D.out = y_out;
  D.P = T;
  D.max_units = D.rows / 16;
  MOE_CUDA(launch_gemv(D, false, true, sms, stream), "down kernel");
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_FORMAT: return "MOE_ERR_UNSUPPORTED_FORMAT";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
    default: return "MOE_ERR_UNKNOWN";
  }
}

const char* moe_last_error(void) { return g_err; }

size_t moe_workspace_bytes(int max_tokens, int n_experts, int top_k, int hidden, int inter) {
  if (max_tokens < 0 || n_experts <= 0 || top_k <= 0 || hidden <= 0 || inter <= 0) return 0;
  if (hidden % 128 != 0 || inter % 128 != 0) return 0;
  return ws_layout(max_tokens, n_experts, top_k, hidden, inter).total;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status s = check_ws(ws, ws_bytes, 256);
  if (s) return s;
  MOE_CUDA(cudaMemsetAsync(ws, 0, 256, stream), "workspace init");
  return ok();
}

moe_status moe_get_device_status(void* ws, size_t ws_bytes, int* device_status,
                                 cudaStream_t stream) {
  moe_status s = check_ws(ws, ws_bytes, 256);
  if (s) return s;
  if (!device_status) return fail(MOE_ERR_INVALID_ARG, "device_status is NULL");
  int v = 0;
  MOE_CUDA(cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, stream), "status read");
  MOE_CUDA(cudaStreamSynchronize(stream), "status sync");
  MOE_CUDA(cudaMemsetAsync(ws, 0, sizeof(int), stream), "status clear");
  *device_status = v;
  return ok();
}

moe_status moe_topk_softmax(const float* logits, int n_tokens, int n_experts, int top_k,
                            int32_t* topk_idx, float* topk_w, cudaStream_t stream) {
  if (n_tokens < 0) return fail(MOE_ERR_INVALID_ARG, "n_tokens=%d < 0", n_tokens);
  if (n_experts < 1 || n_experts > 256)
    return fail(MOE_ERR_INVALID_ARG, "n_experts=%d not in 1..256", n_experts);
  if (top_k < 1 || top_k > 8 || top_k > n_experts)
    return fail(MOE_ERR_INVALID_ARG, "top_k=%d not in 1..min(8, n_experts)", top_k);
  if (n_tokens > 0 && (!logits || !topk_idx || !topk_w))
    return fail(MOE_ERR_INVALID_ARG, "logits/topk_idx/topk_w must not be NULL");
  MOE_CUDA(launch_topk(logits, nullptr, n_tokens, n_experts, top_k, topk_idx, topk_w, nullptr,
                       stream),
           "top-k kernel");
  return ok();
}

moe_status moe_bucket(const int32_t* topk_idx, int n_tokens, int top_k, int n_experts,
                      int32_t* bucket_offsets, int32_t* bucket_perm, cudaStream_t stream) {
  if (n_tokens < 0) return fail(MOE_ERR_INVALID_ARG, "n_tokens=%d < 0", n_tokens);
  if (n_experts < 1 || n_experts > 256)
    return fail(MOE_ERR_INVALID_ARG, "n_experts=%d not in 1..256", n_experts);
  if (top_k < 1 || top_k > 8 || top_k > n_experts)
    return fail(MOE_ERR_INVALID_ARG, "top_k=%d not in 1..min(8, n_experts)", top_k);
  if (!bucket_offsets || (n_tokens > 0 && (!topk_idx || !bucket_perm)))
    return fail(MOE_ERR_INVALID_ARG, "bucket pointers must not be NULL");
  MOE_CUDA(launch_bucket(topk_idx, n_tokens, top_k, n_experts, bucket_offsets, bucket_perm,
                         stream),
           "bucket kernel");
  return ok();
}

moe_status moe_route(const moe_qmatrix* router, const float* logit_bias,
                     const moe_qmatrix* shared_gate, const void* x, int act, int n_tokens,
                     int top_k, float* logits, int32_t* topk_idx, float* topk_w,
                     float* shared_gate_w, int32_t* bucket_offsets, int32_t* bucket_perm,
                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status s;
  if (!router) return fail(MOE_ERR_INVALID_ARG, "router is NULL");
  const int E = router->rows, H = router->cols, T = n_tokens;
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "n_tokens=%d < 0", T);
  if (E < 1 || E > 256) return fail(MOE_ERR_INVALID_ARG, "router rows (experts)=%d not in 1..256", E);
  if (top_k < 1 || top_k > 8 || top_k > E)
    return fail(MOE_ERR_INVALID_ARG, "top_k=%d not in 1..min(8, experts)", top_k);
  if ((s = check_hidden(H))) return s;
  if ((s = check_router_matrix(router, "router", E, H))) return s;
  if (shared_gate && (s = check_router_matrix(shared_gate, "shared_gate", 1, H))) return s;
  if ((s = check_act(act))) return s;
  if (T > 0 && !x) return fail(MOE_ERR_INVALID_ARG, "x is NULL");
  if (x && !aligned16(x)) return fail(MOE_ERR_MISALIGNED, "x not 16-byte aligned");
  if (!bucket_offsets || (T > 0 && (!topk_idx || !topk_w || !bucket_perm)))
    return fail(MOE_ERR_INVALID_ARG, "routing outputs must not be NULL");
  const WsLayout L = ws_layout(T, E, top_k, H, 128);
  if ((s = check_ws(ws, ws_bytes, L.xperm))) return s;
  float* lg = logits ? logits : reinterpret_cast<float*>(wsp(ws, L.logits));
  float* gl = reinterpret_cast<float*>(wsp(ws, L.gate_logit));
  RouterJob R{};
  R.fmt = router->fmt;
  R.q = router->qweight;
  R.s = static_cast<const uint16_t*>(router->scales);
  R.b = static_cast<const uint16_t*>(router->biases);
  if (shared_gate) {
    R.gfmt = shared_gate->fmt;
    R.gq = shared_gate->qweight;
    R.gs = static_cast<const uint16_t*>(shared_gate->scales);
    R.gb = static_cast<const uint16_t*>(shared_gate->biases);
  }
  R.bias = logit_bias;
  R.x = static_cast<const uint16_t*>(x);
  R.f16 = act == MOE_FMT_F16;
  R.T = T;
  R.E = E;
  R.H = H;
  R.logits = lg;
  R.gate_logit = gl;
  MOE_CUDA(launch_router(R, stream), "router kernel");
  MOE_CUDA(launch_topk(lg, shared_gate ? gl : nullptr, T, E, top_k, topk_idx, topk_w,
                       shared_gate ? shared_gate_w : nullptr, stream),
           "top-k kernel");
  MOE_CUDA(launch_bucket(topk_idx, T, top_k, E, bucket_offsets, bucket_perm, stream),
           "bucket kernel");
  return ok();
}

moe_status moe_expert_mlp(const moe_expert_bank* bank, int expert, const void* x, int act,
                          int n_tokens, float* h_out, float* y_out, void* ws, size_t ws_bytes,
                          cudaStream_t stream) {
  moe_status s;
  if ((s = check_bank(bank, "bank"))) return s;
  if ((s = check_act(act))) return s;
  const int T = n_tokens, H = bank->hidden, I = bank->inter;
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "n_tokens=%d < 0", T);
  if (expert < 0 || expert >= bank->n_experts)
    return fail(MOE_ERR_INVALID_ARG, "expert=%d not in 0..%d", expert, bank->n_experts - 1);
  if (T == 0) return ok();
  if (!x || !y_out) return fail(MOE_ERR_INVALID_ARG, "x/y_out is NULL");
  if (!aligned16(x) || !aligned16(y_out) || (h_out && !aligned16(h_out)))
    return fail(MOE_ERR_MISALIGNED, "x/y_out/h_out must be 16-byte aligned");
  const WsLayout L = ws_layout(T, bank->n_experts, 1, H, I);
  if ((s = check_ws(ws, ws_bytes, L.total))) return s;
  s = run_expert_mlp(bank, expert, x, act == MOE_FMT_F16, T, h_out, y_out, ws, L, stream);
  return s ? s : ok();
}

moe_status moe_shared_expert(const moe_expert_bank* shared, const void* x, int act, int n_tokens,
                             float* y_shared, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return moe_expert_mlp(shared, 0, x, act, n_tokens, nullptr, y_shared, ws, ws_bytes, stream);
}

moe_status moe_experts_forward(const moe_expert_bank* experts, const void* x, int act,
                               int n_tokens, int top_k, const int32_t* topk_idx,
                               const float* topk_w, const int32_t* bucket_offsets,
                               const int32_t* bucket_perm, const float* y_shared,
                               const float* shared_gate_w, void* out, int flags, void* ws,
                               size_t ws_bytes, cudaStream_t stream) {
  moe_status s;
  if ((s = check_bank(experts, "experts"))) return s;
  if ((s = check_act(act))) return s;
  const int T = n_tokens, E = experts->n_experts, H = experts->hidden, I = experts->inter;
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "n_tokens=%d < 0", T);
  if (top_k < 1 || top_k > 8 || top_k > E)
    return fail(MOE_ERR_INVALID_ARG, "top_k=%d not in 1..min(8, n_experts)", top_k);
  if (flags & ~MOE_FLAG_FORCE_DECODE) return fail(MOE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  if (T == 0) return ok();
  if (!x || !topk_idx || !topk_w || !bucket_offsets || !bucket_perm || !out)
    return fail(MOE_ERR_INVALID_ARG, "x, routing and out pointers must not be NULL");
  if (!aligned16(x) || !aligned16(out) || (y_shared && !aligned16(y_shared)))
    return fail(MOE_ERR_MISALIGNED, "x/out/y_shared must be 16-byte aligned");
  const WsLayout L = ws_layout(T, E, top_k, H, I);
  if ((s = check_ws(ws, ws_bytes, L.total))) return s;
  const int sms = sm_count();
  const bool f16 = act == MOE_FMT_F16;
  const int P = T * top_k;
  MOE_CUDA(launch_xprep(static_cast<const uint16_t*>(x), T, H, f16,
                        reinterpret_cast<uint16_t*>(wsp(ws, L.xperm)),
                        reinterpret_cast<float*>(wsp(ws, L.xsum)), stream),
           "x prep");
  int* nslots = reinterpret_cast<int*>(wsp(ws, L.nslots));
  int* se = reinterpret_cast<int*>(wsp(ws, L.slot_e));
  int* so = reinterpret_cast<int*>(wsp(ws, L.slot_off));
  int* sc = reinterpret_cast<int*>(wsp(ws, L.slot_cnt));
  int* blist = reinterpret_cast<int*>(wsp(ws, L.blist));
  MOE_CUDA(launch_slots(bucket_offsets, bucket_perm, T, top_k, E, nslots, se, so, sc, blist, stream),
           "slot kernel");
  const int max_slots = E < P ? E : P;
  GemvJob J = bank_job(experts, false);
  J.n_slots = nslots;
  J.slot_expert = se;
  J.slot_off = so;
  J.slot_cnt = sc;
  J.b_row = blist;
  J.B = reinterpret_cast<const uint16_t*>(wsp(ws, L.xperm));
  J.Bsum = reinterpret_cast<const float*>(wsp(ws, L.xsum));
  J.out = reinterpret_cast<float*>(wsp(ws, L.part));
  J.P = P;
  J.max_units = max_slots * (J.rows / 16) * (J.K / J.CK);
  MOE_CUDA(launch_gemv(J, f16, false, sms, stream), "gate/up kernel");
  const int nch = H / J.CK;
  MOE_CUDA(launch_hprep(reinterpret_cast<const float*>(wsp(ws, L.part)), nch, P, I,
                        reinterpret_cast<uint16_t*>(wsp(ws, L.hh)),
                        reinterpret_cast<uint16_t*>(wsp(ws, L.hl)),
                        reinterpret_cast<float*>(wsp(ws, L.hsum)), nullptr, stream),
           "swiglu kernel");
  GemvJob D = bank_job(experts, true);
  D.n_slots = nslots;
  D.slot_expert = se;
  D.slot_off = so;
  D.slot_cnt = sc;
  D.B = reinterpret_cast<const uint16_t*>(wsp(ws, L.hh));
  D.Blo = reinterpret_cast<const uint16_t*>(wsp(ws, L.hl));
  D.Bsum = reinterpret_cast<const float*>(wsp(ws, L.hsum));
  D.out = reinterpret_cast<float*>(wsp(ws, L.y));
  D.out_idx = bucket_perm;
  D.P = P;
  D.max_units = max_slots * (D.rows / 16);
  MOE_CUDA(launch_gemv(D, false, true, sms, stream), "down kernel");
  MOE_CUDA(launch_combine(reinterpret_cast<const float*>(wsp(ws, L.y)), topk_w, top_k, y_shared,
                          shared_gate_w, T, H, f16, static_cast<uint16_t*>(out), stream),
           "combine kernel");
  return ok();
}

moe_status moe_layer_forward(const moe_qmatrix* router, const float* logit_bias,
                             const moe_qmatrix* shared_gate, const moe_expert_bank* experts,
                             const moe_expert_bank* shared, const void* x, int act,
                             int n_tokens, int top_k, void* out, int32_t* topk_idx,
                             float* topk_w, int flags, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
  moe_status s;
  if ((s = check_bank(experts, "experts"))) return s;
  if (shared && (s = check_bank(shared, "shared"))) return s;
  if (!router) return fail(MOE_ERR_INVALID_ARG, "router is NULL");
  const int T = n_tokens, E = experts->n_experts, H = experts->hidden, I = experts->inter;
  if (router->rows != E || router->cols != H)
    return fail(MOE_ERR_INVALID_ARG, "router is [%d, %d], experts need [%d, %d]", router->rows,
                router->cols, E, H);
  if (shared && (shared->hidden != H || shared->inter != I || shared->n_experts != 1))
    return fail(MOE_ERR_INVALID_ARG, "shared bank must be one expert of the experts' shape");
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "n_tokens=%d < 0", T);
  if (top_k < 1 || top_k > 8 || top_k > E)
    return fail(MOE_ERR_INVALID_ARG, "top_k=%d not in 1..min(8, n_experts)", top_k);
  const WsLayout L = ws_layout(T, E, top_k, H, I);
  if ((s = check_ws(ws, ws_bytes, L.total))) return s;
  if (T == 0) return ok();
  int32_t* idx = topk_idx ? topk_idx : reinterpret_cast<int32_t*>(wsp(ws, L.idx));
  float* w = topk_w ? topk_w : reinterpret_cast<float*>(wsp(ws, L.w));
  float* sgw = reinterpret_cast<float*>(wsp(ws, L.sgw));
  int32_t* offs = reinterpret_cast<int32_t*>(wsp(ws, L.offsets));
  int32_t* perm = reinterpret_cast<int32_t*>(wsp(ws, L.perm));
  s = moe_route(router, logit_bias, shared_gate, x, act, T, top_k, nullptr, idx, w,
                shared_gate ? sgw : nullptr, offs, perm, ws, ws_bytes, stream);
  if (s) return s;
  float* ysh = nullptr;
  if (shared) {
    ysh = reinterpret_cast<float*>(wsp(ws, L.ysh));
    s = run_expert_mlp(shared, 0, x, act == MOE_FMT_F16, T, nullptr, ysh, ws, L, stream);
    if (s) return s;
  }
  return moe_experts_forward(experts, x, act, T, top_k, idx, w, offs, perm, ysh,
                             shared && shared_gate ? sgw : nullptr, out, flags, ws, ws_bytes,
                             stream);
}

#define MOE_PACK_PAIR(NAME, FMT, CT)                                                           \
  moe_status moe_pack_##NAME(const CT* codes, int rows, int cols, uint32_t* packed,            \
                             cudaStream_t stream) {                                            \
    if (rows < 0 || cols < 0 || cols % 32 != 0)                                                \
      return fail(MOE_ERR_INVALID_ARG, "pack " #NAME ": rows=%d cols=%d (cols %% 32 == 0)",    \
                  rows, cols);                                                                 \
    if (rows * (long)cols > 0 && (!codes || !packed))                                          \
      return fail(MOE_ERR_INVALID_ARG, "pack " #NAME ": NULL pointer");                        \
    if (packed && !aligned4(packed)) return fail(MOE_ERR_MISALIGNED, "packed not 4-aligned");  \
    MOE_CUDA(launch_pack(FMT, reinterpret_cast<const uint8_t*>(codes), rows, cols, packed,     \
                         stream),                                                              \
             "pack kernel");                                                                   \
    return ok();                                                                               \
  }                                                                                            \
  moe_status moe_unpack_##NAME(const uint32_t* packed, int rows, int cols, CT* codes,          \
                               cudaStream_t stream) {                                          \
    if (rows < 0 || cols < 0 || cols % 32 != 0)                                                \
      return fail(MOE_ERR_INVALID_ARG, "unpack " #NAME ": rows=%d cols=%d (cols %% 32 == 0)",  \
                  rows, cols);                                                                 \
    if (rows * (long)cols > 0 && (!codes || !packed))                                          \
      return fail(MOE_ERR_INVALID_ARG, "unpack " #NAME ": NULL pointer");                      \
    if (packed && !aligned4(packed)) return fail(MOE_ERR_MISALIGNED, "packed not 4-aligned");  \
    MOE_CUDA(launch_unpack(FMT, packed, rows, cols, reinterpret_cast<uint8_t*>(codes), stream), \
             "unpack kernel");                                                                 \
    return ok();                                                                               \
  }

MOE_PACK_PAIR(affine8_g64, MOE_FMT_AFFINE8_G64, uint8_t)
MOE_PACK_PAIR(affine4_g64, MOE_FMT_AFFINE4_G64, uint8_t)
MOE_PACK_PAIR(affine3_g64, MOE_FMT_AFFINE3_G64, uint8_t)
MOE_PACK_PAIR(w4a16_g128, MOE_FMT_W4A16_SYM_G128, int8_t)

moe_status moe_dequant(const moe_qmatrix* m, float* w, cudaStream_t stream) {
  if (!m || !w) return fail(MOE_ERR_INVALID_ARG, "dequant: NULL argument");
  const int f = m->fmt;
  if (f < MOE_FMT_F32 || f > MOE_FMT_W4A16_SYM_G128)
    return fail(MOE_ERR_UNSUPPORTED_FORMAT, "dequant: format %d is not read", f);
  if (m->rows < 0 || m->cols < 0) return fail(MOE_ERR_INVALID_ARG, "dequant: negative shape");
  const int bits = fmt_bits(f);
  if (bits) {
    if (m->cols % 32 != 0 || m->cols % fmt_group(f) != 0)
      return fail(MOE_ERR_INVALID_ARG, "dequant %s: cols=%d must be a multiple of %d", fmt_name(f),
                  m->cols, fmt_group(f) > 32 ? fmt_group(f) : 32);
    if (!m->scales || (f != MOE_FMT_W4A16_SYM_G128 && !m->biases))
      return fail(MOE_ERR_INVALID_ARG, "dequant %s: scales/biases missing", fmt_name(f));
  }
  if (!m->qweight && m->rows * (long)m->cols > 0)
    return fail(MOE_ERR_INVALID_ARG, "dequant: qweight is NULL");
  MOE_CUDA(launch_dequant(f, m->qweight, static_cast<const uint16_t*>(m->scales),
                          static_cast<const uint16_t*>(m->biases), m->rows, m->cols, w, stream),
           "dequant kernel");
  return ok();
}

}  // extern "C"
