// capi.cu -- the extern "C" entry points: argument validation on the host,
// workspace layout, and kernel launches on the caller's stream.
//
// Unsupported widths are refused by name before anything is launched, as the
// loader of "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803"
// refuses any width its kernels do not read (comment "Progress on the 4-bit
// gate", last paragraph).

#include <cuda.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "decode.h"
#include "host.h"
#include "prefill.h"

namespace moe {
int router_ks(int H);

// The driver's cuCtxGetCurrent and cuCtxGetId, reached through the runtime's
// entry-point query (the library links no driver library of its own).
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

cudaError_t ensure_dynamic_smem(const void* func, int bytes) {
  struct Done {
    unsigned long long ctx;
    const void* func;
    int bytes;
  };
  static std::mutex mu;
  static std::vector<Done> done;
  unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (ctx)
    for (const Done& d : done)
      if (d.ctx == ctx && d.func == func && d.bytes >= bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (!ctx) ctx = current_context_id();  // the call above made the primary context current
  if (ctx) {
    for (Done& d : done)
      if (d.ctx == ctx && d.func == func) {
        d.bytes = bytes;
        return cudaSuccess;
      }
    done.push_back(Done{ctx, func, bytes});
  }
  return cudaSuccess;
}

// A second stream with fork and join events, per CUDA context and caller
// stream, for the part of a call that may run beside the work on the
// caller's stream (fork: an event on the caller's stream that the side
// stream waits for; join: the reverse).  Created on first use and kept for
// the life of the process; the events carry no timing.
struct SideStream {
  cudaStream_t s;
  cudaEvent_t fork, join;
  cudaEvent_t xready, tables;  // the layer's early fork: x prepared (side), tables built (caller)
};

cudaError_t side_stream(cudaStream_t user, SideStream* out) {
  struct Entry {
    unsigned long long ctx;
    cudaStream_t user;
    SideStream side;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.ctx == ctx && e.user == user) {
      *out = e.side;
      return cudaSuccess;
    }
  SideStream side{};
  cudaError_t err = cudaStreamCreateWithFlags(&side.s, cudaStreamNonBlocking);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&side.fork, cudaEventDisableTiming);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&side.join, cudaEventDisableTiming);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&side.xready, cudaEventDisableTiming);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&side.tables, cudaEventDisableTiming);
  if (err != cudaSuccess) return err;
  cache.push_back(Entry{ctx ? ctx : current_context_id(), user, side});
  *out = side;
  return cudaSuccess;
}

}  // namespace moe

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
    case MOE_FMT_AFFINE2_G64: return "AFFINE2_G64";
    case MOE_FMT_AFFINE5_G64: return "AFFINE5_G64";
    case MOE_FMT_AFFINE6_G64: return "AFFINE6_G64";
    default: return "unknown";
  }
}

int fmt_bits(int f) {
  switch (f) {
    case MOE_FMT_AFFINE8_G64: return 8;
    case MOE_FMT_AFFINE4_G64: return 4;
    case MOE_FMT_AFFINE3_G64: return 3;
    case MOE_FMT_W4A16_SYM_G128: return 4;
    case MOE_FMT_AFFINE2_G64: return 2;
    case MOE_FMT_AFFINE5_G64: return 5;
    case MOE_FMT_AFFINE6_G64: return 6;
    default: return 0;
  }
}

// Expert formats of the fused decode launch and of the prefill GEMMs; the
// other widths run the launch-per-step decode form (same results as fused).
bool fused_format(int f) {
  return f == MOE_FMT_AFFINE4_G64 || f == MOE_FMT_AFFINE3_G64 || f == MOE_FMT_W4A16_SYM_G128;
}

int fmt_group(int f) { return f == MOE_FMT_W4A16_SYM_G128 ? 128 : 64; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

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

// Format and shape of a bank (either layout).
moe_status check_bank_shape(const moe_expert_bank* b, const char* what) {
  if (!b) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", what);
  const int f = b->fmt;
  if (f != MOE_FMT_AFFINE4_G64 && f != MOE_FMT_AFFINE3_G64 && f != MOE_FMT_W4A16_SYM_G128 &&
      f != MOE_FMT_AFFINE2_G64 && f != MOE_FMT_AFFINE5_G64 && f != MOE_FMT_AFFINE6_G64 &&
      f != MOE_FMT_AFFINE8_G64)
    return fail(MOE_ERR_UNSUPPORTED_FORMAT,
                "%s: expert format %s (%d) is not read by the expert kernels (AFFINE2/3/4/5/6/"
                "8_G64 and W4A16_SYM_G128 are)",
                what, fmt_name(f), f);
  if (b->n_experts <= 0 || b->n_experts > 256)
    return fail(MOE_ERR_INVALID_ARG, "%s: n_experts=%d not in 1..256", what, b->n_experts);
  const int H = b->hidden, I = b->inter;
  const int q = f == MOE_FMT_W4A16_SYM_G128 ? 256 : 128;
  if (H <= 0 || H % q != 0 || I <= 0 || I % q != 0)
    return fail(MOE_ERR_INVALID_ARG, "%s: hidden=%d and inter=%d must be multiples of %d for %s",
                what, H, I, q, fmt_name(f));
  if (I > 512) return fail(MOE_ERR_INVALID_ARG, "%s: inter=%d > 512 unsupported", what, I);
  if (H > 8192) return fail(MOE_ERR_INVALID_ARG, "%s: hidden=%d > 8192 unsupported", what, H);
  return MOE_OK;
}

// A bank the expert kernels read: TILED, two 16-byte aligned buffers.
moe_status check_bank(const moe_expert_bank* b, const char* what) {
  if (moe_status st = check_bank_shape(b, what)) return st;
  if (b->layout != MOE_LAYOUT_TILED)
    return fail(MOE_ERR_INVALID_ARG,
                "%s: layout %d; the expert kernels read TILED banks (moe_repack_bank)", what,
                b->layout);
  if (!b->w13 || !b->w2) return fail(MOE_ERR_INVALID_ARG, "%s: tiled buffer is NULL", what);
  if (!aligned16(b->w13) || !aligned16(b->w2))
    return fail(MOE_ERR_MISALIGNED, "%s: tiled buffers must be 16-byte aligned", what);
  return MOE_OK;
}

// A CANONICAL bank: words 4-byte aligned, scales/biases 2-byte aligned.
moe_status check_canonical(const moe_expert_bank* b, const char* what) {
  if (moe_status st = check_bank_shape(b, what)) return st;
  if (b->layout != MOE_LAYOUT_CANONICAL)
    return fail(MOE_ERR_INVALID_ARG, "%s: layout %d, expected CANONICAL", what, b->layout);
  if (!b->w13 || !b->s13 || !b->w2 || !b->s2)
    return fail(MOE_ERR_INVALID_ARG, "%s: weight or scale pointer is NULL", what);
  if (b->fmt != MOE_FMT_W4A16_SYM_G128 && (!b->b13 || !b->b2))
    return fail(MOE_ERR_INVALID_ARG, "%s: affine format needs biases", what);
  if (!aligned4(b->w13) || !aligned4(b->w2) || !aligned2(b->s13) || !aligned2(b->s2) ||
      (b->b13 && !aligned2(b->b13)) || (b->b2 && !aligned2(b->b2)))
    return fail(MOE_ERR_MISALIGNED, "%s: words need 4-byte, scales/biases 2-byte alignment", what);
  return MOE_OK;
}

// Geometry of w13 (gate/up) and w2 (down) of a TILED bank.
MatGeo geo13(const moe_expert_bank* b) {
  return MatGeo{tile_geo(b->fmt, b->inter, b->hidden, 0), static_cast<const uint8_t*>(b->w13)};
}
MatGeo geo2(const moe_expert_bank* b) {
  return MatGeo{tile_geo(b->fmt, b->inter, b->hidden, 1), static_cast<const uint8_t*>(b->w2)};
}

char* wsp(void* ws, size_t off) { return static_cast<char*>(ws) + off; }

moe_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned16(ws)) return fail(MOE_ERR_MISALIGNED, "workspace not 16-byte aligned");
  if (ws_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, this call needs %zu", ws_bytes, need);
  return MOE_OK;
}

// Engine configuration of one bank in slots 0 (w13) and 1 (w2) (copied to
// 2 and 3): h to the given buffers, y as two k-half planes of yhalf elements.
EngineCfg bank_cfg(const moe_expert_bank* bank, uint16_t* hh, uint16_t* hl, float* hsum,
                   float* hout, float* y, size_t yhalf, int* status) {
  EngineCfg C{};
  C.geo[0] = geo13(bank);
  C.geo[1] = geo2(bank);
  C.geo[2] = C.geo[0];
  C.geo[3] = C.geo[1];
  C.tg[0] = MatTarget{hh, hl, hsum, hout, nullptr, 0};
  C.tg[1] = MatTarget{nullptr, nullptr, nullptr, nullptr, y, yhalf};
  C.tg[2] = C.tg[0];
  C.tg[3] = C.tg[1];
  C.inter = bank->inter;
  C.hidden = bank->hidden;
  C.status = status;
  C.magic_bf16 = 0x43004300u;
  C.magic_f16 = 0x64006400u;
  return C;
}

// Gate/up then down units of one bank over a sub-slot list.  x rows are taken
// by `xrows` (Direct: row = token; Gather: token of a bucket position), h is
// kept at the unit's output rows, y written by `yrows` (Direct or Scatter) as
// two k-half planes (y, y + yhalf).
moe_status run_bank(const moe_expert_bank* bank, const SubSlots& ss, int max_ss, const void* x,
                    bool f16, const float* xsum, int xrows, const int* perm, int k, uint16_t* hh,
                    uint16_t* hl, float* hsum, float* hout, float* y, size_t yhalf, int yrows,
                    int* status, cudaStream_t stream) {
  const int sms = sm_count();
  const int H = bank->hidden, I = bank->inter;
  UnitJob J{};
  J.C = bank_cfg(bank, hh, hl, hsum, hout, y, yhalf, status);
  J.mat = 0;
  J.src = MatSource{static_cast<const uint16_t*>(x), nullptr, xsum, H,
                    sums_ld(J.C.geo[0].t), 0};
  J.rows = xrows;
  J.ss = ss;
  J.perm = perm;
  J.k = k;
  J.max_units = max_ss * (I / 64);
  MOE_CUDA(launch_units(J, f16, sms, stream), "gate/up kernel");
  UnitJob D = J;
  D.mat = 1;
  D.src = MatSource{hh, hl, hsum, h_pitch(I), sums_ld(J.C.geo[1].t), 1};
  D.rows = yrows;
  D.max_units = max_ss * (H / kUnitRows);
  MOE_CUDA(launch_units(D, false, sms, stream), "down kernel");
  return MOE_OK;
}

// One expert (a fixed slot holding every token) over the T rows of x, with
// the given workspace layout: activation sums -> gate/up units (SwiGLU) ->
// down units into the two planes of the workspace's shared-expert output
// (L.ysh); y_out (nullable) receives their sum.
// The prefill form (tcgen05 expert GEMMs) serves T > MOE_DECODE_MAX_TOKENS,
// or any T with MOE_FLAG_FORCE_PREFILL, unless the caller forces the decode
// form or the shape does not fit it.
bool use_prefill(const moe_expert_bank* b, int T, int flags) {
  return (T > MOE_DECODE_MAX_TOKENS || (T > 0 && (flags & MOE_FLAG_FORCE_PREFILL))) &&
         !(flags & MOE_FLAG_FORCE_DECODE) && fused_format(b->fmt) &&
         prefill_smem(geo13(b).t, 0) > 0 && prefill_smem(geo2(b).t, 1) > 0;
}

// MOE_FLAG_FORCE_PREFILL: not with MOE_FLAG_FORCE_DECODE, and only for the
// formats the tensor-core GEMMs read.
moe_status check_force_prefill(const moe_expert_bank* b, int flags) {
  if (!(flags & MOE_FLAG_FORCE_PREFILL)) return MOE_OK;
  if (flags & MOE_FLAG_FORCE_DECODE)
    return fail(MOE_ERR_INVALID_ARG, "MOE_FLAG_FORCE_PREFILL with MOE_FLAG_FORCE_DECODE");
  if (!fused_format(b->fmt))
    return fail(MOE_ERR_UNSUPPORTED_FORMAT,
                "MOE_FLAG_FORCE_PREFILL: the prefill GEMMs do not read %s experts",
                fmt_name(b->fmt));
  return MOE_OK;
}

// The prefill form's activation pass: the per-64-group sums of x (decode
// units) and, for bf16 activations, x's fp16 copy in the workspace (L.xh).
cudaError_t launch_prepare_x(const void* x, bool f16, int T, int H, const TileGeo& g13,
                             float* xsum, void* ws, const WsLayout& L, cudaStream_t stream) {
  if (f16) return launch_xsum(static_cast<const uint16_t*>(x), T, H, true, g13, xsum, stream);
  return launch_xsum_f16(static_cast<const uint16_t*>(x), T, H, g13, xsum,
                         reinterpret_cast<uint16_t*>(wsp(ws, L.xh)), static_cast<int*>(ws),
                         stream);
}

// The shared expert joins the routed experts' prefill launches when both
// take the prefill form with one tiled geometry (same format; the shapes
// are equal by the layer's checks).
bool prefill_pair(const moe_expert_bank* experts, const moe_expert_bank* shared, int T,
                  int flags) {
  return use_prefill(experts, T, flags) && use_prefill(shared, T, flags) &&
         shared->fmt == experts->fmt;
}

// The prefill form's fp16 activation rows: x itself (fp16 activations) or
// its fp16 copy in the workspace (bf16 activations, converted here).
moe_status prefill_act(const void* x, bool f16, int T, int H, void* ws, const WsLayout& L,
                       const uint16_t** out, cudaStream_t stream) {
  if (f16) {
    *out = static_cast<const uint16_t*>(x);
    return MOE_OK;
  }
  uint16_t* xh = reinterpret_cast<uint16_t*>(wsp(ws, L.xh));
  MOE_CUDA(launch_act_f16(static_cast<const uint16_t*>(x), long(T) * H, xh, static_cast<int*>(ws),
                          stream),
           "activation conversion");
  *out = xh;
  return MOE_OK;
}

// One expert of a bank over T tokens in the prefill form: h (fp16) into the
// workspace, y (fp32) straight into y_out.
moe_status run_expert_prefill(const moe_expert_bank* bank, int expert, const void* x, bool f16,
                              int T, float* y_out, void* ws, const WsLayout& L,
                              cudaStream_t stream) {
  const int H = bank->hidden, I = bank->inter;
  const MatGeo g13 = geo13(bank), g2 = geo2(bank);
  const uint16_t* xa = nullptr;
  if (moe_status s = prefill_act(x, f16, T, H, ws, L, &xa, stream)) return s;
  PrefillJob J{};
  J.g = g13.t;
  J.base = g13.base;
  J.fixed_e = expert;
  J.fixed_T = T;
  J.B = xa;
  J.ldB = H;
  J.h = reinterpret_cast<uint16_t*>(wsp(ws, L.sh_hh));
  J.ldh = h_pitch(I);
  J.status = static_cast<int*>(ws);
  MOE_CUDA(launch_prefill(J, 0, sm_count(), stream), "prefill gate/up kernel");
  PrefillJob D = J;
  D.g = g2.t;
  D.base = g2.base;
  D.B = J.h;
  D.ldB = h_pitch(I);
  D.y = y_out;
  D.ldy = H;
  MOE_CUDA(launch_prefill(D, 1, sm_count(), stream), "prefill down kernel");
  return MOE_OK;
}

moe_status run_expert_mlp(const moe_expert_bank* bank, int expert, const void* x, bool f16,
                          int T, float* h_out, float* y_out, void* ws, const WsLayout& L,
                          cudaStream_t stream, int flags = 0) {
  if (!h_out && y_out && use_prefill(bank, T, flags))
    return run_expert_prefill(bank, expert, x, f16, T, y_out, ws, L, stream);
  const int H = bank->hidden;
  float* xsum = reinterpret_cast<float*>(wsp(ws, L.xsum));
  MOE_CUDA(launch_xsum(static_cast<const uint16_t*>(x), T, H, f16, geo13(bank).t, xsum, stream),
           "activation sums");
  const SubSlots ss{nullptr, nullptr, nullptr, nullptr, expert, T};
  float* ysh = reinterpret_cast<float*>(wsp(ws, L.ysh));
  const size_t half = size_t(T) * H;
  moe_status s = run_bank(bank, ss, (T + kMaxTok - 1) / kMaxTok, x, f16, xsum, kRowsDirect,
                          nullptr, 1, reinterpret_cast<uint16_t*>(wsp(ws, L.sh_hh)),
                          reinterpret_cast<uint16_t*>(wsp(ws, L.sh_hl)),
                          reinterpret_cast<float*>(wsp(ws, L.sh_hsum)), h_out, ysh, half,
                          kRowsDirect, static_cast<int*>(ws), stream);
  if (s) return s;
  if (y_out)
    MOE_CUDA(launch_add_planes(ysh, ysh + half, y_out, long(half), stream), "plane sum");
  return MOE_OK;
}

// The routed experts (validated) and, when `shared` is given, the shared
// expert folded into the same prefill launches (its output into L.ysh, which
// is then the combine's shared row): see prefill_pair.
moe_status experts_run(const moe_expert_bank* experts, const moe_expert_bank* shared,
                       const void* x, bool f16, int T, int top_k, const int32_t* topk_idx,
                       const float* topk_w, const int32_t* bucket_offsets,
                       const int32_t* bucket_perm, const float* y_shared,
                       const float* shared_gate_w, void* out, int flags, void* ws,
                       const WsLayout& L, cudaStream_t stream,
                       const SideStream* early = nullptr) {
  moe_status s;
  const int E = experts->n_experts, H = experts->hidden, I = experts->inter;
  const bool rb = (flags & MOE_FLAG_ROUND_BF16) != 0;
  if (use_prefill(experts, T, flags)) {
    // Experts with more than kPfLight assignments: tiles of up to kPfTile
    // bucket positions through the tensor-core GEMMs (second y plane set to
    // 0); the others: sub-slots of 8 through the decode units.  One combine
    // over the two y planes.
    float* y = reinterpret_cast<float*>(wsp(ws, L.y));
    const size_t yhalf = size_t(T) * top_k * H;
    int* nt = reinterpret_cast<int*>(wsp(ws, L.pt_n));
    int* te = reinterpret_cast<int*>(wsp(ws, L.pt_e));
    int* to = reinterpret_cast<int*>(wsp(ws, L.pt_off));
    int* tc = reinterpret_cast<int*>(wsp(ws, L.pt_cnt));
    int* nss = reinterpret_cast<int*>(wsp(ws, L.nss));
    int* se = reinterpret_cast<int*>(wsp(ws, L.ss_e));
    int* so = reinterpret_cast<int*>(wsp(ws, L.ss_off));
    int* sc = reinterpret_cast<int*>(wsp(ws, L.ss_cnt));
    const MatGeo g13 = geo13(experts), g2 = geo2(experts);
    float* xsum = reinterpret_cast<float*>(wsp(ws, L.xsum));
    const uint16_t* xa =
        f16 ? static_cast<const uint16_t*>(x) : reinterpret_cast<uint16_t*>(wsp(ws, L.xh));
    // the light experts (decode units, y planes 0 and 1 of their own rows, h
    // rows of their own bucket positions) on a side stream, beside the
    // tensor-core GEMMs of the others; joined before the combine
    SideStream side{};
    if (early) {
      // moe_layer_forward already built the tables with the bucket sort and
      // started the side stream on x (launch_prepare_x): hand it the tables
      side = *early;
      MOE_CUDA(cudaEventRecord(side.tables, stream), "tables event");
      MOE_CUDA(cudaStreamWaitEvent(side.s, side.tables, 0), "tables wait");
    } else {
      MOE_CUDA(launch_subslots_pair(bucket_offsets, E, kPfLight, SubslotTable{nt, te, to, tc},
                                    kPfTile, SubslotTable{nss, se, so, sc}, kMaxTok, stream),
               "tile and sub-slot kernel");
      MOE_CUDA(launch_prepare_x(x, f16, T, H, g13.t, xsum, ws, L, stream), "activation sums");
      MOE_CUDA(side_stream(stream, &side), "side stream");
      MOE_CUDA(cudaEventRecord(side.fork, stream), "fork event");
      MOE_CUDA(cudaStreamWaitEvent(side.s, side.fork, 0), "fork wait");
    }
    {
      const SubSlots ss{nss, se, so, sc, 0, 0};
      s = run_bank(experts, ss, int(max_subslots(T, E, top_k)), x, f16, xsum, kRowsGather,
                   bucket_perm, top_k, reinterpret_cast<uint16_t*>(wsp(ws, L.hh)),
                   reinterpret_cast<uint16_t*>(wsp(ws, L.hl)),
                   reinterpret_cast<float*>(wsp(ws, L.hsum)), nullptr, y, yhalf, kRowsScatter,
                   static_cast<int*>(ws), side.s);
      if (s) return s;
    }
    MOE_CUDA(cudaEventRecord(side.join, side.s), "join event");
    if (early) MOE_CUDA(cudaStreamWaitEvent(stream, side.xready, 0), "x wait");
    PrefillJob J{};
    J.g = g13.t;
    J.base = g13.base;
    J.n_tiles = nt;
    J.te = te;
    J.toff = to;
    J.tcnt = tc;
    J.B = xa;
    J.ldB = H;
    J.gather = 1;
    J.perm = bucket_perm;
    J.k = top_k;
    J.h = reinterpret_cast<uint16_t*>(wsp(ws, L.hh));  // fp16 h rows of the tiled experts
    J.ldh = h_pitch(I);
    J.status = static_cast<int*>(ws);
    if (shared) {
      J.sh_base = geo13(shared).base;
      J.sh_T = T;
      J.sh_B = xa;
      J.sh_h = reinterpret_cast<uint16_t*>(wsp(ws, L.sh_hh));
      y_shared = reinterpret_cast<float*>(wsp(ws, L.ysh));
    }
    MOE_CUDA(launch_prefill(J, 0, sm_count(), stream), "prefill gate/up kernel");
    PrefillJob D = J;
    D.g = g2.t;
    D.base = g2.base;
    D.B = J.h;
    D.ldB = h_pitch(I);
    D.gather = 0;
    D.y = y;
    D.ldy = H;
    D.scatter = 1;
    if (shared) {
      D.sh_base = geo2(shared).base;
      D.sh_B = J.sh_h;
      D.sh_h = nullptr;
      D.sh_y = const_cast<float*>(y_shared);
    }
    MOE_CUDA(launch_prefill(D, 1, sm_count(), stream), "prefill down kernel");
    MOE_CUDA(cudaStreamWaitEvent(stream, side.join, 0), "join wait");
    CombineArgs C{};
    C.y = y;
    C.yhalf = yhalf;
    C.w = topk_w;
    C.ysh = y_shared;
    C.ysh2 = nullptr;
    C.sg = shared_gate_w;
    C.out = static_cast<uint16_t*>(out);
    C.T = T;
    C.k = top_k;
    C.H = H;
    C.f16 = f16;
    C.round_bf16 = rb;
    C.idx = topk_idx;  // the tiled experts' y sits in plane 0 alone
    C.offsets = bucket_offsets;
    C.one_plane_max = kPfLight;
    MOE_CUDA(launch_combine(C, stream), "combine kernel");
    return ok();
  }
  float* xsum = reinterpret_cast<float*>(wsp(ws, L.xsum));
  MOE_CUDA(launch_xsum(static_cast<const uint16_t*>(x), T, H, f16, geo13(experts).t, xsum,
                       stream),
           "activation sums");
  int* nss = reinterpret_cast<int*>(wsp(ws, L.nss));
  int* se = reinterpret_cast<int*>(wsp(ws, L.ss_e));
  int* so = reinterpret_cast<int*>(wsp(ws, L.ss_off));
  int* sc = reinterpret_cast<int*>(wsp(ws, L.ss_cnt));
  MOE_CUDA(launch_subslots(bucket_offsets, E, nss, se, so, sc, stream), "sub-slot kernel");
  const SubSlots ss{nss, se, so, sc, 0, 0};
  float* y = reinterpret_cast<float*>(wsp(ws, L.y));
  const size_t yhalf = size_t(T) * top_k * H;
  s = run_bank(experts, ss, int(max_subslots(T, E, top_k)), x, f16, xsum, kRowsGather,
               bucket_perm, top_k, reinterpret_cast<uint16_t*>(wsp(ws, L.hh)),
               reinterpret_cast<uint16_t*>(wsp(ws, L.hl)),
               reinterpret_cast<float*>(wsp(ws, L.hsum)), nullptr, y, yhalf, kRowsScatter,
               static_cast<int*>(ws), stream);
  if (s) return s;
  CombineArgs C{};
  C.y = y;
  C.yhalf = yhalf;
  C.w = topk_w;
  C.ysh = y_shared;
  C.ysh2 = nullptr;
  C.sg = shared_gate_w;
  C.out = static_cast<uint16_t*>(out);
  C.T = T;
  C.k = top_k;
  C.H = H;
  C.f16 = f16;
  C.round_bf16 = rb;
  MOE_CUDA(launch_combine(C, stream), "combine kernel");
  return ok();
}

// moe_route's argument checks (router, gate, activations, sizes).
moe_status route_check(const moe_qmatrix* router, const moe_qmatrix* shared_gate, const void* x,
                       int act, int T, int top_k) {
  moe_status s;
  const int E = router->rows, H = router->cols;
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
  return MOE_OK;
}

// The prefill form's tile and sub-slot tables, built by the bucket launch.
struct PrefillTables {
  int split;
  SubslotTable A;
  int run_a;
  SubslotTable B;
  int run_b;
};

// moe_route's launches (checked arguments) on workspace layout L: router and
// top-k, then the bucket sort (with `tables`, also the prefill tables).
moe_status route_run(const moe_qmatrix* router, const float* logit_bias,
                     const moe_qmatrix* shared_gate, const void* x, bool f16, int T, int top_k,
                     float* logits, int32_t* topk_idx, float* topk_w, float* shared_gate_w,
                     int32_t* bucket_offsets, int32_t* bucket_perm, bool rb, void* ws,
                     const WsLayout& L, const PrefillTables* tables, cudaStream_t stream) {
  const int E = router->rows, H = router->cols;
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
  R.f16 = f16;
  R.T = T;
  R.E = E;
  R.H = H;
  R.logits = lg;
  R.gate_logit = gl;
  R.round_bf16 = rb;
  R.part = T > MOE_DECODE_MAX_TOKENS ? reinterpret_cast<float*>(wsp(ws, L.rpart)) : nullptr;
  R.split = T > MOE_DECODE_MAX_TOKENS ? reinterpret_cast<uint16_t*>(wsp(ws, L.rsplit)) : nullptr;
  MOE_CUDA(launch_router_topk(R, top_k, topk_idx, topk_w, shared_gate_w, rb, stream),
           "router and top-k kernels");
  if (tables)
    MOE_CUDA(launch_bucket_tables(topk_idx, T, top_k, E, bucket_offsets, bucket_perm,
                                  tables->split, tables->A, tables->run_a, tables->B,
                                  tables->run_b, stream),
             "bucket and table kernel");
  else
    MOE_CUDA(launch_bucket(topk_idx, T, top_k, E, bucket_offsets, bucket_perm, stream),
             "bucket kernel");
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
    case MOE_ERR_RANGE: return "MOE_ERR_RANGE";
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
  moe_status s = check_ws(ws, ws_bytes, kCtlBytes);
  if (s) return s;
  MOE_CUDA(cudaMemsetAsync(ws, 0, kCtlBytes, stream), "workspace init");
  return ok();
}

moe_status moe_workspace_set_wait_limit(void* ws, size_t ws_bytes, unsigned limit_us,
                                        cudaStream_t stream) {
  moe_status s = check_ws(ws, ws_bytes, kCtlBytes);
  if (s) return s;
  if (limit_us > 0x7FFFFFFFu)
    return fail(MOE_ERR_INVALID_ARG, "limit_us=%u exceeds 2^31 - 1", limit_us);
  MOE_CUDA(launch_store_word(static_cast<int*>(ws) + kCtlWaitLimit, int(limit_us), stream),
           "wait-limit store");
  return ok();
}

moe_status moe_get_device_status(void* ws, size_t ws_bytes, int* device_status,
                                 cudaStream_t stream) {
  moe_status s = check_ws(ws, ws_bytes, kCtlBytes);
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
                       false, stream),
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
                     int flags, void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status s;
  if (!router) return fail(MOE_ERR_INVALID_ARG, "router is NULL");
  if (flags & ~MOE_FLAG_ROUND_BF16) return fail(MOE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  const int E = router->rows, H = router->cols, T = n_tokens;
  if ((s = route_check(router, shared_gate, x, act, T, top_k))) return s;
  if (!bucket_offsets || (T > 0 && (!topk_idx || !topk_w || !bucket_perm)))
    return fail(MOE_ERR_INVALID_ARG, "routing outputs must not be NULL");
  const WsLayout L = ws_layout(T, E, top_k, H, 128);
  // the logits, and above the decode sizes the router's k-slice sums and
  // bf16 parts
  if ((s = check_ws(ws, ws_bytes,
                    T > MOE_DECODE_MAX_TOKENS ? L.rsplit + 2 * router_split_elems(T, E, H) : L.idx)))
    return s;
  s = route_run(router, logit_bias, shared_gate, x, act == MOE_FMT_F16, T, top_k, logits,
                topk_idx, topk_w, shared_gate_w, bucket_offsets, bucket_perm,
                (flags & MOE_FLAG_ROUND_BF16) != 0, ws, L, nullptr, stream);
  return s ? s : ok();
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
  if (flags & ~(MOE_FLAG_FORCE_DECODE | MOE_FLAG_FORCE_PREFILL | MOE_FLAG_ROUND_BF16))
    return fail(MOE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  if ((s = check_force_prefill(experts, flags))) return s;
  if (T == 0) return ok();
  if (!x || !topk_idx || !topk_w || !bucket_offsets || !bucket_perm || !out)
    return fail(MOE_ERR_INVALID_ARG, "x, routing and out pointers must not be NULL");
  if (!aligned16(x) || !aligned16(out) || (y_shared && !aligned16(y_shared)))
    return fail(MOE_ERR_MISALIGNED, "x/out/y_shared must be 16-byte aligned");
  const WsLayout L = ws_layout(T, E, top_k, H, I);
  if ((s = check_ws(ws, ws_bytes, L.total))) return s;
  return experts_run(experts, nullptr, x, act == MOE_FMT_F16, T, top_k, topk_idx, topk_w,
                     bucket_offsets, bucket_perm, y_shared, shared_gate_w, out, flags, ws, L,
                     stream);
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
  if (flags &
      ~(MOE_FLAG_FORCE_DECODE | MOE_FLAG_FORCE_PREFILL | MOE_FLAG_UNFUSED | MOE_FLAG_ROUND_BF16))
    return fail(MOE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  if ((s = check_force_prefill(experts, flags))) return s;
  const bool rb = (flags & MOE_FLAG_ROUND_BF16) != 0;
  if (!(flags & (MOE_FLAG_UNFUSED | MOE_FLAG_FORCE_PREFILL)) && T <= MOE_DECODE_MAX_TOKENS &&
      fused_format(experts->fmt) &&
      (!shared || fused_format(shared->fmt))) {
    // validate what moe_route / moe_experts_forward would, then one launch
    if ((s = check_hidden(H))) return s;
    if ((s = check_router_matrix(router, "router", E, H))) return s;
    if (shared_gate && (s = check_router_matrix(shared_gate, "shared_gate", 1, H))) return s;
    if ((s = check_act(act))) return s;
    if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "x/out is NULL");
    if (!aligned16(x) || !aligned16(out))
      return fail(MOE_ERR_MISALIGNED, "x/out must be 16-byte aligned");
    const bool f16 = act == MOE_FMT_F16;
    DecodeArgs A{};
    A.R.fmt = router->fmt;
    A.R.q = router->qweight;
    A.R.s = static_cast<const uint16_t*>(router->scales);
    A.R.b = static_cast<const uint16_t*>(router->biases);
    if (shared_gate) {
      A.R.gfmt = shared_gate->fmt;
      A.R.gq = shared_gate->qweight;
      A.R.gs = static_cast<const uint16_t*>(shared_gate->scales);
      A.R.gb = static_cast<const uint16_t*>(shared_gate->biases);
    }
    A.R.bias = logit_bias;
    A.R.x = static_cast<const uint16_t*>(x);
    A.R.f16 = f16;
    A.R.T = T;
    A.R.E = E;
    A.R.H = H;
    A.R.round_bf16 = rb;
    int* status = static_cast<int*>(ws);
    uint16_t* hh = reinterpret_cast<uint16_t*>(wsp(ws, L.hh));
    uint16_t* hl = reinterpret_cast<uint16_t*>(wsp(ws, L.hl));
    float* hsum = reinterpret_cast<float*>(wsp(ws, L.hsum));
    uint16_t* shh = reinterpret_cast<uint16_t*>(wsp(ws, L.sh_hh));
    uint16_t* shl = reinterpret_cast<uint16_t*>(wsp(ws, L.sh_hl));
    float* shsum = reinterpret_cast<float*>(wsp(ws, L.sh_hsum));
    float* xsum = reinterpret_cast<float*>(wsp(ws, L.xsum));
    float* y = reinterpret_cast<float*>(wsp(ws, L.y));
    float* ysh = reinterpret_cast<float*>(wsp(ws, L.ysh));
    A.C = bank_cfg(experts, hh, hl, hsum, nullptr, y, size_t(T) * top_k * H, status);
    if (shared) {
      A.C.geo[2] = geo13(shared);
      A.C.geo[3] = geo2(shared);
    }
    A.C.tg[2] = MatTarget{shh, shl, shsum, nullptr, nullptr, 0};
    A.C.tg[3] = MatTarget{nullptr, nullptr, nullptr, nullptr, ysh, size_t(T) * H};
    const int ldx = sums_ld(A.C.geo[0].t), ldh = sums_ld(A.C.geo[1].t);
    A.src[0] = MatSource{A.R.x, nullptr, xsum, H, ldx, 0};
    A.src[1] = MatSource{hh, hl, hsum, h_pitch(I), ldh, 1};
    A.src[2] = A.src[0];
    A.src[3] = MatSource{shh, shl, shsum, h_pitch(I), ldh, 1};
    A.k = top_k;
    A.has_shared = shared ? 1 : 0;
    A.KS = router_ks(H);
    A.R.logits = reinterpret_cast<float*>(wsp(ws, L.logits));
    A.R.gate_logit = reinterpret_cast<float*>(wsp(ws, L.gate_logit));
    A.user_idx = topk_idx;
    A.user_w = topk_w;
    A.out = static_cast<uint16_t*>(out);
    A.ctrl = status;
    const EnginePlan P = decode_plan(A);
    if (P.S < 2)
      return fail(MOE_ERR_INVALID_ARG,
                  "shape needs %d-byte operand buffers and %d-byte stages; they do not fit in "
                  "shared memory",
                  P.OB, P.SB);
    MOE_CUDA(launch_decode(A, experts->fmt, shared ? shared->fmt : experts->fmt, sm_count(),
                           stream),
             "fused decode kernel");
    return ok();
  }
  int32_t* idx = topk_idx ? topk_idx : reinterpret_cast<int32_t*>(wsp(ws, L.idx));
  float* w = topk_w ? topk_w : reinterpret_cast<float*>(wsp(ws, L.w));
  float* sgw = reinterpret_cast<float*>(wsp(ws, L.sgw));
  int32_t* offs = reinterpret_cast<int32_t*>(wsp(ws, L.offsets));
  int32_t* perm = reinterpret_cast<int32_t*>(wsp(ws, L.perm));
  const int ef = flags & (MOE_FLAG_FORCE_DECODE | MOE_FLAG_FORCE_PREFILL | MOE_FLAG_ROUND_BF16);
  const bool fold = shared && prefill_pair(experts, shared, T, ef);
  if (use_prefill(experts, T, ef) && (!shared || fold)) {
    // The prefill form in one pass over the workspace layout L: the side
    // stream starts on x (sums and fp16 copy) at once, beside the routing,
    // whose bucket launch also builds the tile and sub-slot tables; the
    // experts then run with the shared expert folded into their launches.
    if ((s = route_check(router, shared_gate, x, act, T, top_k))) return s;
    if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "x/out is NULL");
    if (!aligned16(out)) return fail(MOE_ERR_MISALIGNED, "out must be 16-byte aligned");
    const bool f16 = act == MOE_FMT_F16;
    SideStream side{};
    MOE_CUDA(side_stream(stream, &side), "side stream");
    MOE_CUDA(cudaEventRecord(side.fork, stream), "fork event");
    MOE_CUDA(cudaStreamWaitEvent(side.s, side.fork, 0), "fork wait");
    MOE_CUDA(launch_prepare_x(x, f16, T, H, geo13(experts).t,
                              reinterpret_cast<float*>(wsp(ws, L.xsum)), ws, L, side.s),
             "activation sums");
    MOE_CUDA(cudaEventRecord(side.xready, side.s), "x event");
    const PrefillTables tb{
        kPfLight,
        SubslotTable{reinterpret_cast<int*>(wsp(ws, L.pt_n)), reinterpret_cast<int*>(wsp(ws, L.pt_e)),
                     reinterpret_cast<int*>(wsp(ws, L.pt_off)),
                     reinterpret_cast<int*>(wsp(ws, L.pt_cnt))},
        kPfTile,
        SubslotTable{reinterpret_cast<int*>(wsp(ws, L.nss)), reinterpret_cast<int*>(wsp(ws, L.ss_e)),
                     reinterpret_cast<int*>(wsp(ws, L.ss_off)),
                     reinterpret_cast<int*>(wsp(ws, L.ss_cnt))},
        kMaxTok};
    s = route_run(router, logit_bias, shared_gate, x, f16, T, top_k, nullptr, idx, w,
                  shared_gate ? sgw : nullptr, offs, perm, (ef & MOE_FLAG_ROUND_BF16) != 0, ws, L,
                  &tb, stream);
    if (s) return s;
    s = experts_run(experts, fold ? shared : nullptr, x, f16, T, top_k, idx, w, offs, perm,
                    nullptr, fold && shared_gate ? sgw : nullptr, out, ef, ws, L, stream, &side);
    return s ? s : ok();
  }
  s = moe_route(router, logit_bias, shared_gate, x, act, T, top_k, nullptr, idx, w,
                shared_gate ? sgw : nullptr, offs, perm, flags & MOE_FLAG_ROUND_BF16, ws, ws_bytes,
                stream);
  if (s) return s;
  float* ysh = nullptr;
  if (shared) {
    ysh = reinterpret_cast<float*>(wsp(ws, L.ysh));
    s = run_expert_mlp(shared, 0, x, act == MOE_FMT_F16, T, nullptr, ysh, ws, L, stream, flags);
    if (s) return s;
  }
  return moe_experts_forward(experts, x, act, T, top_k, idx, w, offs, perm, ysh,
                             shared && shared_gate ? sgw : nullptr, out, ef, ws, ws_bytes, stream);
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
MOE_PACK_PAIR(affine2_g64, MOE_FMT_AFFINE2_G64, uint8_t)
MOE_PACK_PAIR(affine5_g64, MOE_FMT_AFFINE5_G64, uint8_t)
MOE_PACK_PAIR(affine6_g64, MOE_FMT_AFFINE6_G64, uint8_t)

size_t moe_tiled_bytes(int fmt, int n_experts, int inter, int hidden, int which) {
  moe_expert_bank b{};
  b.fmt = fmt;
  b.n_experts = n_experts;
  b.inter = inter;
  b.hidden = hidden;
  if (check_bank_shape(&b, "tiled_bytes") || (which != 0 && which != 1)) return 0;
  return size_t(tile_geo(fmt, inter, hidden, which).expert_bytes) * size_t(n_experts);
}

moe_status moe_repack_bank(const moe_expert_bank* canonical, void* w13_tiled, void* w2_tiled,
                           cudaStream_t stream) {
  if (moe_status st = check_canonical(canonical, "repack: canonical bank")) return st;
  if (!w13_tiled || !w2_tiled) return fail(MOE_ERR_INVALID_ARG, "repack: tiled buffer is NULL");
  if (!aligned16(w13_tiled) || !aligned16(w2_tiled))
    return fail(MOE_ERR_MISALIGNED, "repack: tiled buffers must be 16-byte aligned");
  const moe_expert_bank& b = *canonical;
  const bool aff = b.fmt != MOE_FMT_W4A16_SYM_G128;
  MOE_CUDA(launch_repack(tile_geo(b.fmt, b.inter, b.hidden, 0), b.n_experts,
                         static_cast<const uint32_t*>(b.w13), static_cast<const uint16_t*>(b.s13),
                         aff ? static_cast<const uint16_t*>(b.b13) : nullptr,
                         static_cast<uint8_t*>(w13_tiled), stream),
           "repack w13");
  MOE_CUDA(launch_repack(tile_geo(b.fmt, b.inter, b.hidden, 1), b.n_experts,
                         static_cast<const uint32_t*>(b.w2), static_cast<const uint16_t*>(b.s2),
                         aff ? static_cast<const uint16_t*>(b.b2) : nullptr,
                         static_cast<uint8_t*>(w2_tiled), stream),
           "repack w2");
  return ok();
}

moe_status moe_unrepack_bank(const moe_expert_bank* tiled, void* w13, void* s13, void* b13,
                             void* w2, void* s2, void* b2, cudaStream_t stream) {
  if (moe_status st = check_bank(tiled, "unrepack: tiled bank")) return st;
  const bool aff = tiled->fmt != MOE_FMT_W4A16_SYM_G128;
  if (!w13 || !s13 || !w2 || !s2 || (aff && (!b13 || !b2)))
    return fail(MOE_ERR_INVALID_ARG, "unrepack: output pointer is NULL");
  if (!aligned4(w13) || !aligned4(w2) || !aligned2(s13) || !aligned2(s2) ||
      (aff && (!aligned2(b13) || !aligned2(b2))))
    return fail(MOE_ERR_MISALIGNED, "unrepack: words need 4-byte, scales 2-byte alignment");
  const moe_expert_bank& b = *tiled;
  MOE_CUDA(launch_unrepack(tile_geo(b.fmt, b.inter, b.hidden, 0), b.n_experts,
                           static_cast<const uint8_t*>(b.w13), static_cast<uint32_t*>(w13),
                           static_cast<uint16_t*>(s13), aff ? static_cast<uint16_t*>(b13) : nullptr,
                           stream),
           "unrepack w13");
  MOE_CUDA(launch_unrepack(tile_geo(b.fmt, b.inter, b.hidden, 1), b.n_experts,
                           static_cast<const uint8_t*>(b.w2), static_cast<uint32_t*>(w2),
                           static_cast<uint16_t*>(s2), aff ? static_cast<uint16_t*>(b2) : nullptr,
                           stream),
           "unrepack w2");
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Routing without a caller workspace (moe_route_static).  Some callers cannot
// hand the library memory: a caller that owns no device allocator of its own
// (a plain C host application driving the layer through this ABI), or one that
// must not allocate once its serving loop runs (cudaMalloc synchronises the
// device and may fail under memory pressure).  For them the router's one
// scratch buffer -- the fp32 logits and shared-gate logits between the router
// kernel and the top-k kernel -- lives in this file-scope device array.
// Nothing in it has to start at zero: every element a call reads was written
// earlier in the same call.  There is one copy of the array per CUDA context
// (it belongs to the module loaded into that context), so calls that overlap
// in time within one context (two streams, two host threads) race on it.
namespace {

constexpr int kStaticRouteMaxLogits = 32 * 256;  // T * E of at most 32 tokens x 256 experts
constexpr int kStaticRouteMaxTokens = 32;        // shared-gate logits
__device__ __align__(256) float g_static_route_scratch[kStaticRouteMaxLogits +
                                                       kStaticRouteMaxTokens];

// The array's device address in the current context.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress once per context (the first call in a context does
// this synchronous runtime query, so it should come before any stream
// capture) and cached under the context's id: after cudaDeviceReset, or in a
// driver-API context, the module is loaded again and the array may sit
// elsewhere.
moe_status static_route_scratch(float** out) {
  struct Entry {
    unsigned long long ctx;
    float* addr;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (ctx)
    for (const Entry& c : cache)
      if (c.ctx == ctx) {
        *out = c.addr;
        return MOE_OK;
      }
  void* p = nullptr;
  MOE_CUDA(cudaGetSymbolAddress(&p, g_static_route_scratch), "cudaGetSymbolAddress");
  if (!ctx) ctx = current_context_id();  // the lookup made the primary context current
  if (ctx) cache.push_back(Entry{ctx, static_cast<float*>(p)});
  *out = static_cast<float*>(p);
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_route_static(const moe_qmatrix* router, const float* logit_bias,
                            const moe_qmatrix* shared_gate, const void* x, int act,
                            int n_tokens, int top_k, int32_t* topk_idx, float* topk_w,
                            float* shared_gate_w, int32_t* bucket_offsets, int32_t* bucket_perm,
                            cudaStream_t stream) {
  moe_status s;
  if (!router) return fail(MOE_ERR_INVALID_ARG, "router is NULL");
  const int E = router->rows, H = router->cols, T = n_tokens;
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "n_tokens=%d < 0", T);
  if (E < 1 || E > 256) return fail(MOE_ERR_INVALID_ARG, "router rows (experts)=%d not in 1..256", E);
  if (top_k < 1 || top_k > 8 || top_k > E)
    return fail(MOE_ERR_INVALID_ARG, "top_k=%d not in 1..min(8, experts)", top_k);
  if (T > kStaticRouteMaxTokens || long(T) * E > kStaticRouteMaxLogits)
    return fail(MOE_ERR_WORKSPACE,
                "moe_route_static: n_tokens=%d x experts=%d exceeds its static scratch of %d "
                "logits (at most %d tokens); use moe_route with a workspace",
                T, E, kStaticRouteMaxLogits, kStaticRouteMaxTokens);
  if ((s = check_hidden(H))) return s;
  if ((s = check_router_matrix(router, "router", E, H))) return s;
  if (shared_gate && (s = check_router_matrix(shared_gate, "shared_gate", 1, H))) return s;
  if ((s = check_act(act))) return s;
  if (T > 0 && !x) return fail(MOE_ERR_INVALID_ARG, "x is NULL");
  if (x && !aligned16(x)) return fail(MOE_ERR_MISALIGNED, "x not 16-byte aligned");
  if (!bucket_offsets || (T > 0 && (!topk_idx || !topk_w || !bucket_perm)))
    return fail(MOE_ERR_INVALID_ARG, "routing outputs must not be NULL");
  float* scratch = nullptr;
  if ((s = static_route_scratch(&scratch))) return s;
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
  R.logits = scratch;
  R.gate_logit = scratch + kStaticRouteMaxLogits;
  MOE_CUDA(launch_router(R, stream), "router kernel");
  MOE_CUDA(launch_topk(R.logits, shared_gate ? R.gate_logit : nullptr, T, E, top_k, topk_idx,
                       topk_w, shared_gate ? shared_gate_w : nullptr, false, stream),
           "top-k kernel");
  MOE_CUDA(launch_bucket(topk_idx, T, top_k, E, bucket_offsets, bucket_perm, stream),
           "bucket kernel");
  return ok();
}

moe_status moe_dequant(const moe_qmatrix* m, float* w, cudaStream_t stream) {
  if (!m || !w) return fail(MOE_ERR_INVALID_ARG, "dequant: NULL argument");
  const int f = m->fmt;
  if (f < MOE_FMT_F32 || f > MOE_FMT_AFFINE6_G64)
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
