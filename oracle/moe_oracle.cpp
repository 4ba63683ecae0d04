// moe_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU reference of the routed-expert MoE layer over
// low-bit affine-quantised weights.  Only the test suite, the package's
// smoke() check and bench.py's CPU-baseline and reference legs may load it; the
// library's GPU path never does, and this file shares no code, header,
// table or constant with the CUDA sources.
//
// Sources followed (cited by page title and section):
//  [803-run]   "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803",
//              Description, "What I want to run": MLX affine in groups of 64,
//              routed experts 3-bit, everything else 4-bit, router and
//              shared-expert gate 8-bit.
//  [803-gate]  same issue, comment "Progress on the 4-bit gate", paragraph
//              "What is in it": fp32 logits over the experts and the shared
//              gate row, top-k by logit with ties to the lower id, weights
//              exp(l - l_top) over the k, the shared expert as a further slot
//              weighted by sigmoid(gate), the slots' fma sum, experts with a
//              SwiGLU epilogue (gate and up interleaved per group).
//  [803-fp64]  same issue, "Affine experts at other widths": an FP64
//              reference per projection class.
//  [803-widen] same issue, comment "The 3-bit width is up as #972": 3-bit
//              codes rewritten as 4-bit words give the same results.
//  [w4a16]     "Sage-1.5-W4A16" model card, "Model details" and "Recipe":
//              int4 symmetric weights, group 128, no zero point,
//              pack-quantized compressed-tensors export.
//  [1329]      "Sage-A1.5 (qwen3_5 MoE 35B-A3B) on the XPU backend ... #1329",
//              Proposal: 256 experts with top-8, hidden 2048, grouped MoE.
//
// The pages give prose only (no formulas or listings).  Where they are
// silent the plainest reading is taken and stated at the function.
//
// Parity status: every function here is pinned by the CPU tests (format
// round trips and hand-derived words, exact dequant, brute-force top-k,
// closed-form softmax, bucketing invariants, one-expert layer = dense
// SwiGLU MLP through numpy, width-widening equality, bf16 rounding against
// torch's conversion, fp32 combine cases that only the fused multiply-add,
// the slot order or the shared slot's place decide, 2/5/6-bit streams over
// every code at every position, exact dequantisation at every width, the
// same codes at every width giving the same weights and layer output, the
// layer's bf16 rounding-chain option on hand-worked bf16 closed forms).  None
// is unpinned.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <numeric>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---------------------------------------------------------------------------
// Format codes of this oracle (its own numbering; the Python wrapper maps
// names to them).
enum OFmt {
  O_F32 = 0,          // plain fp32 values
  O_BF16 = 1,         // bfloat16 bit patterns
  O_F16 = 2,          // IEEE binary16 bit patterns
  O_AFFINE8_G64 = 3,  // MLX affine 8-bit, group 64: w = s*q + b
  O_AFFINE4_G64 = 4,  // MLX affine 4-bit, group 64
  O_AFFINE3_G64 = 5,  // MLX affine 3-bit, group 64 (LSB-first bit stream)
  O_W4A16_G128 = 6,   // compressed-tensors int4 symmetric, group 128: w = s*q
  O_AFFINE2_G64 = 7,  // MLX affine at the other widths the loader reads [803-fp64]
  O_AFFINE5_G64 = 8,
  O_AFFINE6_G64 = 9,
};

int code_bits(int fmt) {
  switch (fmt) {
    case O_AFFINE8_G64: return 8;
    case O_AFFINE4_G64: return 4;
    case O_AFFINE3_G64: return 3;
    case O_W4A16_G128: return 4;
    case O_AFFINE2_G64: return 2;
    case O_AFFINE5_G64: return 5;
    case O_AFFINE6_G64: return 6;
    default: return 0;
  }
}

int group_size(int fmt) {
  switch (fmt) {
    case O_AFFINE8_G64:
    case O_AFFINE4_G64:
    case O_AFFINE3_G64:
    case O_AFFINE2_G64:
    case O_AFFINE5_G64:
    case O_AFFINE6_G64: return 64;
    case O_W4A16_G128: return 128;
    default: return 0;
  }
}

bool is_quantized(int fmt) { return code_bits(fmt) != 0; }

// 32-bit words per row of packed codes.
long words_per_row(int fmt, long cols) { return cols * code_bits(fmt) / 32; }

// IEEE binary16 -> double, straight from the encoding: 1 sign bit, 5 exponent
// bits (bias 15), 10 fraction bits; exponent 0 is subnormal, 31 is inf/NaN.
double half_bits_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = std::ldexp((double)f, -24);
  } else if (e == 31) {
    v = f ? std::nan("") : INFINITY;
  } else {
    v = std::ldexp(1.0 + f / 1024.0, e - 15);
  }
  return sign ? -v : v;
}

// bfloat16 -> double: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
double bf16_bits_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int f = b & 0x7f;
  double v;
  if (e == 0) {
    v = std::ldexp((double)f, -133);
  } else if (e == 255) {
    v = f ? std::nan("") : INFINITY;
  } else {
    v = std::ldexp(1.0 + f / 128.0, e - 127);
  }
  return sign ? -v : v;
}

// One code out of a packed row.  Affine 8/4/2-bit and W4A16: 32/bits codes
// per little-endian uint32, code i of a word at bits [bits*i, bits*i + bits).
// Affine 3/5/6-bit (widths that do not divide 32): the row is one LSB-first
// bit stream; code c occupies stream bits [bits*c, bits*c + bits), which may
// straddle two words.  (Both rules are the same stream for widths dividing
// 32; the pages state the 3-bit stream, and 5/6-bit are read the same way.)
bool stream_width(int fmt) { return 32 % code_bits(fmt) != 0; }

uint32_t get_code(int fmt, const uint32_t* row_words, long c) {
  int bits = code_bits(fmt);
  if (stream_width(fmt)) {
    uint32_t v = 0;
    for (int i = 0; i < bits; ++i) {
      long bit = (long)bits * c + i;
      uint32_t b = (row_words[bit / 32] >> (bit % 32)) & 1u;
      v |= b << i;
    }
    return v;
  }
  long per = 32 / bits;
  uint32_t w = row_words[c / per];
  return (w >> (bits * (c % per))) & ((1u << bits) - 1u);
}

void put_code(int fmt, uint32_t* row_words, long c, uint32_t v) {
  int bits = code_bits(fmt);
  if (stream_width(fmt)) {
    for (int i = 0; i < bits; ++i) {
      long bit = (long)bits * c + i;
      uint32_t b = (v >> i) & 1u;
      row_words[bit / 32] |= b << (bit % 32);
    }
    return;
  }
  long per = 32 / bits;
  row_words[c / per] |= (v & ((1u << bits) - 1u)) << (bits * (c % per));
}

// Dequantise one packed/dense matrix [rows, cols] into doubles.
// Affine (MLX): w = scale * q + bias per group of 64 along cols [803-run].
// W4A16 (compressed-tensors pack-quantized) [w4a16]: the stored nibble u is
// offset binary, q = u - 8 in -8..7, w = scale * q (symmetric, no zero point).
// In fp64 each product and sum here is exact: an fp16 scale has 11
// significant bits and a code at most 8.
int dequant(int fmt, long rows, long cols, const void* q, const uint16_t* s,
            const uint16_t* b, double* out) {
  if (fmt == O_F32) {
    const float* f = (const float*)q;
    for (long i = 0; i < rows * cols; ++i) out[i] = (double)f[i];
    return 0;
  }
  if (fmt == O_BF16 || fmt == O_F16) {
    const uint16_t* h = (const uint16_t*)q;
    for (long i = 0; i < rows * cols; ++i)
      out[i] = fmt == O_BF16 ? bf16_bits_to_double(h[i]) : half_bits_to_double(h[i]);
    return 0;
  }
  if (!is_quantized(fmt)) return -1;
  int G = group_size(fmt);
  if (cols % G != 0 || cols % 32 != 0) return -2;
  long wpr = words_per_row(fmt, cols);
  long gpr = cols / G;
  const uint32_t* words = (const uint32_t*)q;
  for (long r = 0; r < rows; ++r) {
    const uint32_t* rw = words + r * wpr;
    for (long c = 0; c < cols; ++c) {
      double scale = half_bits_to_double(s[r * gpr + c / G]);
      double code = (double)get_code(fmt, rw, c);
      if (fmt == O_W4A16_G128) {
        out[r * cols + c] = scale * (code - 8.0);
      } else {
        double bias = half_bits_to_double(b[r * gpr + c / G]);
        out[r * cols + c] = scale * code + bias;
      }
    }
  }
  return 0;
}

// Bytes of one stored matrix (codes/values only).
long value_bytes(int fmt, long rows, long cols) {
  if (fmt == O_F32) return rows * cols * 4;
  if (fmt == O_BF16 || fmt == O_F16) return rows * cols * 2;
  return rows * words_per_row(fmt, cols) * 4;
}

long group_count(int fmt, long rows, long cols) {
  if (!is_quantized(fmt)) return 0;
  return rows * (cols / group_size(fmt));
}

bool has_bias(int fmt) { return is_quantized(fmt) && fmt != O_W4A16_G128; }

// Ordering for top-k [803-gate]: larger logit first; equal logits go to the
// lower expert id.  The pages test a NaN row without saying where NaN ranks;
// the reading here: NaN ranks below every number (also below -inf), NaNs
// among themselves by id.
bool ranks_before(double la, int ia, double lb, int ib) {
  bool na = std::isnan(la), nb = std::isnan(lb);
  if (na != nb) return nb;
  if (!na && la != lb) return la > lb;
  return ia < ib;
}

double silu(double a) { return a / (1.0 + std::exp(-a)); }

// y[t, r] = sum_c W[r, c] * x[t, c]
void matvec_rows(const double* W, long rows, long cols, const double* x, long T,
                 double* y) {
  for (long t = 0; t < T; ++t)
    for (long r = 0; r < rows; ++r) {
      double acc = 0.0;
      const double* wr = W + r * cols;
      const double* xt = x + t * cols;
      for (long c = 0; c < cols; ++c) acc += wr[c] * xt[c];
      y[t * rows + r] = acc;
    }
}

// bf16 from fp32: round to nearest, ties to even; a NaN becomes the quiet NaN
// 0x7FC0.  bf16 is the top half of the fp32 encoding, so widening is exact.
static uint16_t f32_to_bf16_rne(float v) {
  uint32_t u;
  std::memcpy(&u, &v, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
  const uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
  return uint16_t((u + bias) >> 16);
}

static float bf16_to_f32(uint16_t b) {
  const uint32_t u = uint32_t(b) << 16;
  float v;
  std::memcpy(&v, &u, 4);
  return v;
}

// An fp64 value through the engine's storage types: first fp32, then bf16.
double via_f32_bf16(double v) { return (double)bf16_to_f32(f32_to_bf16_rne((float)v)); }

}  // namespace

extern "C" {

int oracle_abi_version() { return 2; }

int oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

int oracle_code_bits(int fmt) { return code_bits(fmt); }
int oracle_group_size(int fmt) { return group_size(fmt); }
long oracle_value_bytes(int fmt, long rows, long cols) { return value_bytes(fmt, rows, cols); }

// Pack integer codes [rows, cols] into the format's words.  Affine codes are
// unsigned (0 .. 2^bits - 1); W4A16 codes are signed q in -8..7 and are stored
// as u = q + 8 [w4a16].  Returns 0, or a negative value on a code out of range.
int oracle_pack(int fmt, long rows, long cols, const int32_t* codes, uint32_t* words) {
  if (!is_quantized(fmt) || cols % 32 != 0) return -1;
  long wpr = words_per_row(fmt, cols);
  std::memset(words, 0, sizeof(uint32_t) * rows * wpr);
  int bits = code_bits(fmt);
  for (long r = 0; r < rows; ++r)
    for (long c = 0; c < cols; ++c) {
      int32_t v = codes[r * cols + c];
      if (fmt == O_W4A16_G128) {
        if (v < -8 || v > 7) return -2;
        v += 8;
      } else if (v < 0 || v >= (1 << bits)) {
        return -2;
      }
      put_code(fmt, words + r * wpr, c, (uint32_t)v);
    }
  return 0;
}

int oracle_unpack(int fmt, long rows, long cols, const uint32_t* words, int32_t* codes) {
  if (!is_quantized(fmt) || cols % 32 != 0) return -1;
  long wpr = words_per_row(fmt, cols);
  for (long r = 0; r < rows; ++r)
    for (long c = 0; c < cols; ++c) {
      int32_t v = (int32_t)get_code(fmt, words + r * wpr, c);
      if (fmt == O_W4A16_G128) v -= 8;
      codes[r * cols + c] = v;
    }
  return 0;
}

int oracle_dequant(int fmt, long rows, long cols, const void* q, const uint16_t* s,
                   const uint16_t* b, double* out) {
  return dequant(fmt, rows, cols, q, s, b, out);
}

// Activations (bf16 or fp16 bit patterns, or fp32) -> double.
int oracle_act_to_double(int fmt, long n, const void* x, double* out) {
  if (fmt == O_F32) {
    for (long i = 0; i < n; ++i) out[i] = (double)((const float*)x)[i];
  } else if (fmt == O_BF16) {
    for (long i = 0; i < n; ++i) out[i] = bf16_bits_to_double(((const uint16_t*)x)[i]);
  } else if (fmt == O_F16) {
    for (long i = 0; i < n; ++i) out[i] = half_bits_to_double(((const uint16_t*)x)[i]);
  } else {
    return -1;
  }
  return 0;
}

int oracle_fp16_to_double(long n, const uint16_t* h, double* out) {
  for (long i = 0; i < n; ++i) out[i] = half_bits_to_double(h[i]);
  return 0;
}

// Router logits [803-gate]: l[t, e] = sum_h W_r[e, h] * x[t, h] + bias[e].
// W_r is fp32, bf16 or affine-8 g64 (the 3-bit checkpoint's 8-bit router,
// [803-run]).  bias (nullable) is a per-expert logit offset.
// bf16_rows: the dequantised rows are first rounded to bf16 (through fp32),
// as the engine stores its 8-bit router rows after loading them [803-gate].
static int router_logits(int wfmt, long E, long H, const void* wq, const uint16_t* ws,
                         const uint16_t* wb, const float* bias, long T, const double* x,
                         double* logits, bool bf16_rows) {
  std::vector<double> W((size_t)E * H);
  int rc = dequant(wfmt, E, H, wq, ws, wb, W.data());
  if (rc) return rc;
  if (bf16_rows)
    for (double& v : W) v = via_f32_bf16(v);
  matvec_rows(W.data(), E, H, x, T, logits);
  if (bias)
    for (long t = 0; t < T; ++t)
      for (long e = 0; e < E; ++e) logits[t * E + e] += (double)bias[e];
  return 0;
}

int oracle_router_logits(int wfmt, long E, long H, const void* wq, const uint16_t* ws,
                         const uint16_t* wb, const float* bias, long T,
                         const double* x, double* logits) {
  return router_logits(wfmt, E, H, wq, ws, wb, bias, T, x, logits, false);
}

// Top-k and routing weights [803-gate].  Experts are ordered by (logit desc,
// id asc) and the first k become slots 0..k-1.  The weights are exp(l - l_top)
// over the k; read as normalised over the k (a softmax over the selected
// experts), so w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0).
int oracle_topk(long T, long E, long k, const double* logits, int32_t* idx, double* w) {
  if (k < 1 || k > E) return -1;
  std::vector<int> order(E);
  for (long t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    std::iota(order.begin(), order.end(), 0);
    std::sort(order.begin(), order.end(),
              [&](int a, int b) { return ranks_before(l[a], a, l[b], b); });
    double top = l[order[0]];
    double den = 0.0;
    for (long j = 0; j < k; ++j) den += std::exp(l[order[j]] - top);
    for (long j = 0; j < k; ++j) {
      idx[t * k + j] = order[j];
      w[t * k + j] = std::exp(l[order[j]] - top) / den;
    }
  }
  return 0;
}

// Shared-expert gate [803-gate]: g_t = sum_h w_g[h] x[t, h] over the shared
// gate row (affine-8 g64, bf16 or fp32), weight s_t = sigmoid(g_t).
// bf16_chain: the gate row is rounded to bf16 like the router rows, and the
// weight becomes bf16(sigmoid(bf16(g))) [803-gate] (sigmoid in fp64).
static int shared_gate(int gfmt, long H, const void* gq, const uint16_t* gs,
                       const uint16_t* gb, long T, const double* x, double* logit,
                       double* sg, bool bf16_chain) {
  std::vector<double> g((size_t)H);
  int rc = dequant(gfmt, 1, H, gq, gs, gb, g.data());
  if (rc) return rc;
  if (bf16_chain)
    for (double& v : g) v = via_f32_bf16(v);
  for (long t = 0; t < T; ++t) {
    double acc = 0.0;
    for (long h = 0; h < H; ++h) acc += g[h] * x[t * H + h];
    if (logit) logit[t] = acc;
    if (bf16_chain)
      sg[t] = via_f32_bf16(1.0 / (1.0 + std::exp(-via_f32_bf16(acc))));
    else
      sg[t] = 1.0 / (1.0 + std::exp(-acc));
  }
  return 0;
}

int oracle_shared_gate(int gfmt, long H, const void* gq, const uint16_t* gs,
                       const uint16_t* gb, long T, const double* x, double* logit,
                       double* sg) {
  return shared_gate(gfmt, H, gq, gs, gb, T, x, logit, sg, false);
}

// One expert's SwiGLU MLP [803-gate] on dequantised weights.  w13 holds the
// gate rows (0 .. I-1) followed by the up rows (I .. 2I-1) of [2I, H]; w2 is
// the down projection [H, I].  a = Wg x, b = Wu x, h = silu(a) * b, y = Wd h.
// The pages name a SwiGLU epilogue without writing it out; silu(gate) * up is
// the plain reading.  h and y are outputs (h nullable).
int oracle_expert_mlp(int fmt, long I, long H, const void* w13, const uint16_t* s13,
                      const uint16_t* b13, const void* w2, const uint16_t* s2,
                      const uint16_t* b2, long T, const double* x, double* h_out,
                      double* y) {
  std::vector<double> W13((size_t)2 * I * H), W2((size_t)H * I);
  int rc = dequant(fmt, 2 * I, H, w13, s13, b13, W13.data());
  if (rc) return rc;
  rc = dequant(fmt, H, I, w2, s2, b2, W2.data());
  if (rc) return rc;
  std::vector<double> ab((size_t)T * 2 * I), h((size_t)T * I);
  matvec_rows(W13.data(), 2 * I, H, x, T, ab.data());
  for (long t = 0; t < T; ++t)
    for (long j = 0; j < I; ++j) {
      double a = ab[t * 2 * I + j];
      double b = ab[t * 2 * I + I + j];
      h[t * I + j] = silu(a) * b;
    }
  matvec_rows(W2.data(), H, I, h.data(), T, y);
  if (h_out) std::memcpy(h_out, h.data(), sizeof(double) * T * I);
  return 0;
}

// Down projection alone (per-projection checks [803-fp64]): y = Wd h.
int oracle_down(int fmt, long H, long I, const void* w2, const uint16_t* s2,
                const uint16_t* b2, long T, const double* h, double* y) {
  std::vector<double> W2((size_t)H * I);
  int rc = dequant(fmt, H, I, w2, s2, b2, W2.data());
  if (rc) return rc;
  matvec_rows(W2.data(), H, I, h, T, y);
  return 0;
}

// Token -> expert bucketing (grouped MoE, [1329]): a counting sort of the
// assignment ids a = t*k + j by expert, stable (ascending a inside a bucket).
// counts[E], offsets[E+1] (exclusive prefix sum), perm[T*k], and the active
// experts (count > 0) in ascending id.
int oracle_bucket(long T, long k, long E, const int32_t* idx, int32_t* counts,
                  int32_t* offsets, int32_t* perm, int32_t* active, int32_t* n_active) {
  for (long e = 0; e < E; ++e) counts[e] = 0;
  for (long a = 0; a < T * k; ++a) {
    int e = idx[a];
    if (e < 0 || e >= E) return -1;
    counts[e]++;
  }
  offsets[0] = 0;
  for (long e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> cursor(offsets, offsets + E);
  for (long a = 0; a < T * k; ++a) perm[cursor[idx[a]]++] = (int32_t)a;
  int32_t n = 0;
  for (long e = 0; e < E; ++e)
    if (counts[e] > 0) active[n++] = (int32_t)e;
  *n_active = n;
  return 0;
}

// The whole layer [803-gate]:
//   logits -> top-k -> weights; shared gate; every active expert's SwiGLU MLP
//   on its tokens; out[t] = sum_j w[t,j] * y[t,j] + s_t * y_shared[t],
// kept in fp64 (the GPU output is compared before its final cast).
//
// Experts: bank of E experts in one format, w13 [E][2I][H], w2 [E][H][I]
// (codes/values contiguous per expert; scales/biases likewise).
// The shared expert (nullable: shared_w13 == NULL) uses its own format; the
// shared gate row (nullable) is affine-8/bf16/fp32.  With no shared gate the
// shared expert is added with weight 1.
// idx_override (nullable) replaces the computed top-k indices (weights are
// then the softmax of this oracle's own logits over those indices); used
// when fp32 logits on the GPU resolve a near tie differently.
// round_bf16 selects the engine's bf16 rounding chain for the routing inputs
// (router and gate rows, slot weights, shared weight); the logits, the
// experts and the weighted sum stay fp64 and out stays unrounded.
struct LayerArgs {
  long T, E, k, H, I;
  const double* x;                 // [T][H]
  int router_fmt;
  const void* router_q; const uint16_t* router_s; const uint16_t* router_b;
  const float* logit_bias;         // [E] or NULL
  int expert_fmt;
  const void* w13; const uint16_t* s13; const uint16_t* b13;
  const void* w2; const uint16_t* s2; const uint16_t* b2;
  int shared_fmt;
  const void* sh_w13; const uint16_t* sh_s13; const uint16_t* sh_b13;
  const void* sh_w2; const uint16_t* sh_s2; const uint16_t* sh_b2;
  int gate_fmt;
  const void* gate_q; const uint16_t* gate_s; const uint16_t* gate_b;
  const int32_t* idx_override;     // [T][k] or NULL
  // outputs (all nullable except out)
  double* logits;                  // [T][E]
  int32_t* idx;                    // [T][k]
  double* w;                       // [T][k]
  double* sg;                      // [T]
  double* y_slots;                 // [T][k][H]
  double* y_shared;                // [T][H]
  double* out;                     // [T][H]
  // 1: the engine's bf16 rounding chain [803-gate] -- router and gate rows
  // rounded to bf16, slot weights bf16(w), shared weight
  // bf16(sigmoid(bf16(g))); 0: weights and gate kept exact.
  int round_bf16;
};

int oracle_moe_layer(const LayerArgs* A) {
  const long T = A->T, E = A->E, k = A->k, H = A->H, I = A->I;
  const bool rb = A->round_bf16 != 0;
  std::vector<double> logits((size_t)T * E);
  int rc = router_logits(A->router_fmt, E, H, A->router_q, A->router_s, A->router_b,
                         A->logit_bias, T, A->x, logits.data(), rb);
  if (rc) return rc;
  std::vector<int32_t> idx((size_t)T * k);
  std::vector<double> w((size_t)T * k);
  rc = oracle_topk(T, E, k, logits.data(), idx.data(), w.data());
  if (rc) return rc;
  if (A->idx_override) {
    for (long t = 0; t < T; ++t) {
      const double* l = logits.data() + t * E;
      const int32_t* o = A->idx_override + t * k;
      double top = l[o[0]];
      double den = 0.0;
      for (long j = 0; j < k; ++j) den += std::exp(l[o[j]] - top);
      for (long j = 0; j < k; ++j) {
        idx[t * k + j] = o[j];
        w[t * k + j] = std::exp(l[o[j]] - top) / den;
      }
    }
  }
  if (rb)
    for (double& v : w) v = via_f32_bf16(v);
  std::vector<double> sg((size_t)T, 1.0);
  if (A->gate_q) {
    rc = shared_gate(A->gate_fmt, H, A->gate_q, A->gate_s, A->gate_b, T, A->x, nullptr,
                     sg.data(), rb);
    if (rc) return rc;
  }

  // Per-expert strides inside the bank.
  const long w13_bytes = value_bytes(A->expert_fmt, 2 * I, H);
  const long w2_bytes = value_bytes(A->expert_fmt, H, I);
  const long g13 = group_count(A->expert_fmt, 2 * I, H);
  const long g2 = group_count(A->expert_fmt, H, I);
  const bool hb = has_bias(A->expert_fmt);

  std::vector<double> yslots((size_t)T * k * H, 0.0);
  std::vector<int> active;
  for (long e = 0; e < E; ++e) {
    bool used = false;
    for (long a = 0; a < T * k && !used; ++a) used = idx[a] == e;
    if (used) active.push_back((int)e);
  }
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long ai = 0; ai < (long)active.size(); ++ai) {
    const int e = active[ai];
    std::vector<long> slots;
    for (long a = 0; a < T * k; ++a)
      if (idx[a] == e) slots.push_back(a);
    const long n = (long)slots.size();
    std::vector<double> xe((size_t)n * H), ye((size_t)n * H);
    for (long i = 0; i < n; ++i)
      std::memcpy(&xe[i * H], A->x + (slots[i] / k) * H, sizeof(double) * H);
    int r = oracle_expert_mlp(
        A->expert_fmt, I, H, (const char*)A->w13 + e * w13_bytes,
        A->s13 ? A->s13 + e * g13 : nullptr, hb ? A->b13 + e * g13 : nullptr,
        (const char*)A->w2 + e * w2_bytes, A->s2 ? A->s2 + e * g2 : nullptr,
        hb ? A->b2 + e * g2 : nullptr, n, xe.data(), nullptr, ye.data());
    if (r) {
#pragma omp critical
      err = r;
    }
    for (long i = 0; i < n; ++i)
      std::memcpy(&yslots[slots[i] * H], &ye[i * H], sizeof(double) * H);
  }
  if (err) return err;

  std::vector<double> ysh((size_t)T * H, 0.0);
  if (A->sh_w13) {
    rc = oracle_expert_mlp(A->shared_fmt, I, H, A->sh_w13, A->sh_s13, A->sh_b13, A->sh_w2,
                           A->sh_s2, A->sh_b2, T, A->x, nullptr, ysh.data());
    if (rc) return rc;
  }
  for (long t = 0; t < T; ++t)
    for (long h = 0; h < H; ++h) {
      double acc = 0.0;
      for (long j = 0; j < k; ++j) acc += w[t * k + j] * yslots[(t * k + j) * H + h];
      if (A->sh_w13) acc += sg[t] * ysh[t * H + h];
      A->out[t * H + h] = acc;
    }
  if (A->logits) std::memcpy(A->logits, logits.data(), sizeof(double) * T * E);
  if (A->idx) std::memcpy(A->idx, idx.data(), sizeof(int32_t) * T * k);
  if (A->w) std::memcpy(A->w, w.data(), sizeof(double) * T * k);
  if (A->sg) std::memcpy(A->sg, sg.data(), sizeof(double) * T);
  if (A->y_slots) std::memcpy(A->y_slots, yslots.data(), sizeof(double) * T * k * H);
  if (A->y_shared) std::memcpy(A->y_shared, ysh.data(), sizeof(double) * T * H);
  return 0;
}

// ---------------------------------------------------------------------------
// fp32 values rounded to bf16 (nearest, ties to even) and widened back.
int oracle_round_bf16(long n, const float* in, float* out) {
  for (long i = 0; i < n; ++i) out[i] = bf16_to_f32(f32_to_bf16_rne(in[i]));
  return 0;
}

// The combine in the engine's own precision [803-gate]: the slots' fma sum in
// fp32 -- slot order, the shared slot last -- rounded once to bf16.  Given the
// slots' outputs and weights as fp32 values, every bit of the result is fixed
// by IEEE arithmetic, so a device combine fed the same inputs can be compared
// byte for byte.  Rounding to bf16 is to nearest, ties to even; a NaN becomes
// the quiet NaN 0x7FC0.
//   y [T*k][H], w [T][k], ysh [T][H] (nullable), sg [T] (nullable: weight 1),
//   out [T][H] bf16 bit patterns.
int oracle_combine_f32(long T, long k, long H, const float* y, const float* w,
                       const float* ysh, const float* sg, uint16_t* out) {
  if (T < 0 || k < 1 || H < 0) return -1;
  for (long t = 0; t < T; ++t)
    for (long h = 0; h < H; ++h) {
      float acc = 0.f;
      for (long j = 0; j < k; ++j) acc = std::fmaf(w[t * k + j], y[(t * k + j) * H + h], acc);
      if (ysh) acc = std::fmaf(sg ? sg[t] : 1.f, ysh[t * H + h], acc);
      out[t * H + h] = f32_to_bf16_rne(acc);
    }
  return 0;
}

// The engine's rounding chain for the shared slot [803-gate]: slot weights
// rounded to bf16, the shared slot weighted by bf16(sigmoid(bf16(g)))
// (the sigmoid evaluated in fp64 on the bf16 gate logit).
int oracle_chain_gate_weight(long T, const float* g, float* s) {
  for (long t = 0; t < T; ++t) {
    const double gb = bf16_to_f32(f32_to_bf16_rne(g[t]));
    s[t] = bf16_to_f32(f32_to_bf16_rne(float(1.0 / (1.0 + std::exp(-gb)))));
  }
  return 0;
}

}  // extern "C"
