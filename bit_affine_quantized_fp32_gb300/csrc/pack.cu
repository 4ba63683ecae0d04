// pack.cu -- pack / unpack / dequantise for the quantised storage formats.
//
// Formats: MLX affine 8/4/3-bit in groups of 64 ("qwen3_5_moe on native CUDA
// with 3-bit routed experts ... #803", Description: "stored as MLX affine in
// groups of 64"; 3-bit routed experts, 8-bit router and shared gate) with
// w = scale * q + bias; compressed-tensors pack-quantized int4 symmetric,
// group 128 ("Sage-1.5-W4A16", Model details) with w = scale * q, stored as
// the offset-binary nibble q + 8.  Codes sit LSB-first in little-endian
// uint32 words; a 3-bit row is one bit stream (code c at bits [3c, 3c+3)).

#include "common.cuh"
#include "kernels.h"
#include "tiled.cuh"

namespace moe {

namespace {

__host__ __device__ inline int fmt_bits(int fmt) {
  switch (fmt) {
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

// widths whose codes straddle word boundaries (a row is one bit stream)
__host__ __device__ inline bool fmt_stream(int fmt) {
  const int b = fmt_bits(fmt);
  return b == 3 || b == 5 || b == 6;
}

// one thread per packed word
__global__ void k_pack(int fmt, const uint8_t* __restrict__ codes, int rows, int cols,
                       uint32_t* __restrict__ packed) {
  const int bits = fmt_bits(fmt);
  const long wpr = long(cols) * bits / 32;
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= long(rows) * wpr) return;
  const long r = i / wpr, j = i - r * wpr;
  const uint8_t* row = codes + r * cols;
  uint32_t v = 0;
  if (fmt_stream(fmt)) {
    for (int b = 0; b < 32; ++b) {
      const long s = j * 32 + b;
      const uint32_t code = row[s / bits];
      v |= ((code >> (s % bits)) & 1u) << b;
    }
  } else {
    const int per = 32 / bits;
    const uint32_t mask = (1u << bits) - 1u;
    for (int q = 0; q < per; ++q) {
      uint32_t code = row[j * per + q];
      if (fmt == MOE_FMT_W4A16_SYM_G128) code = uint32_t(int(int8_t(code)) + 8);
      v |= (code & mask) << (bits * q);
    }
  }
  packed[i] = v;
}

__device__ __forceinline__ uint32_t get_code(int fmt, const uint32_t* row, long c) {
  const int bits = fmt_bits(fmt);
  if (fmt_stream(fmt)) {
    const long s = long(bits) * c;
    const long w = s >> 5;
    const int b = int(s & 31);
    uint32_t v = row[w] >> b;
    if (b > 32 - bits) v |= row[w + 1] << (32 - b);
    return v & ((1u << bits) - 1u);
  }
  const int per = 32 / bits;
  return (row[c / per] >> (bits * (c % per))) & ((1u << bits) - 1u);
}

// one thread per code
__global__ void k_unpack(int fmt, const uint32_t* __restrict__ packed, int rows, int cols,
                         uint8_t* __restrict__ codes) {
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= long(rows) * cols) return;
  const long r = i / cols, c = i - r * cols;
  const long wpr = long(cols) * fmt_bits(fmt) / 32;
  uint32_t v = get_code(fmt, packed + r * wpr, c);
  if (fmt == MOE_FMT_W4A16_SYM_G128) v = uint32_t(int(v) - 8) & 0xFFu;
  codes[i] = uint8_t(v);
}

// one thread per element
__global__ void k_dequant(int fmt, const void* __restrict__ q, const uint16_t* __restrict__ s,
                          const uint16_t* __restrict__ b, int rows, int cols,
                          float* __restrict__ w) {
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= long(rows) * cols) return;
  if (fmt == MOE_FMT_F32) {
    w[i] = static_cast<const float*>(q)[i];
    return;
  }
  if (fmt == MOE_FMT_BF16 || fmt == MOE_FMT_F16) {
    w[i] = act_to_float(static_cast<const uint16_t*>(q)[i], fmt == MOE_FMT_F16);
    return;
  }
  const long r = i / cols, c = i - r * cols;
  const long wpr = long(cols) * fmt_bits(fmt) / 32;
  const uint32_t code = get_code(fmt, static_cast<const uint32_t*>(q) + r * wpr, c);
  const int G = fmt == MOE_FMT_W4A16_SYM_G128 ? 128 : 64;
  const long gi = r * (cols / G) + c / G;
  const float sc = half_bits_to_float(s[gi]);
  if (fmt == MOE_FMT_W4A16_SYM_G128) {
    w[i] = sc * float(int(code) - 8);
  } else {
    w[i] = fmaf(sc, float(code), half_bits_to_float(b[gi]));
  }
}

// ---- kernel-tiled layout (geometry in tiled.cuh) --------------------------

// Where code (row r, column k) of expert e sits in a tiled buffer.
struct TiledPos {
  long long block;  // byte offset of its (w, G) code block
  int lane;         // fragment lane g*4 + t
  int widx;         // word W0..W3 of that lane
  int nib;          // code index inside the word
};

__device__ __forceinline__ void tiled_rowpos(const TileGeo& g, int r, int& blk, int& w, int& sub) {
  if (g.down) {
    blk = r / 128;
    w = (r % 128) / 16;
  } else if (r < g.inter) {
    blk = r / 64;
    w = (r % 64) / 16;
  } else {
    blk = (r - g.inter) / 64;
    w = 4 + ((r - g.inter) % 64) / 16;
  }
  sub = r % 16;
}

__device__ __forceinline__ long long tiled_item(const TileGeo& g, int e, int blk, int c) {
  return (long long)e * g.expert_bytes + (long long)(blk * g.nch + c) * g.item_bytes;
}

__device__ __forceinline__ TiledPos tiled_pos(const TileGeo& g, int e, int r, int k) {
  int blk, w, sub;
  tiled_rowpos(g, r, blk, w, sub);
  const int c = k / g.CK, kk = k % g.CK;
  const int G = kk / 64, t = (kk % 64) / 16, half = (kk % 16) / 8;
  TiledPos p;
  p.block = tiled_item(g, e, blk, c) + (long long)(w * g.ng + G) * tiled_cb(g.fmt);
  p.lane = (sub & 7) * 4 + t;
  p.widx = (sub >> 3) * 2 + half;
  p.nib = tiled_nib(k % 8);
  return p;
}

// one thread per (expert, item, tile w, group G, lane): the lane's four words
__global__ void k_repack_codes(TileGeo g, int E, const uint32_t* __restrict__ wc,
                               uint8_t* __restrict__ out) {
  const long long n = (long long)E * g.nblk * g.nch * 8 * g.ng * 32;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  long long q = i;
  const int lane = int(q % 32); q /= 32;
  const int G = int(q % g.ng); q /= g.ng;
  const int w = int(q % 8); q /= 8;
  const int c = int(q % g.nch); q /= g.nch;
  const int blk = int(q % g.nblk); q /= g.nblk;
  const int e = int(q);
  const int gq = lane >> 2, t = lane & 3;
  const int r0 = tiled_row(g, blk, w) + gq;
  const int k0 = c * g.CK + 64 * G + 16 * t;
  const long wpr = long(g.K) * fmt_bits(g.fmt) / 32;
  // low 4 bits of each code as the nibble words W0..W3, the rest per format
  uint32_t W[4], HW[4] = {0, 0, 0, 0}, P5 = 0, P6[2] = {0, 0};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = r0 + (j >> 1) * 8;
    const uint32_t* row = wc + ((long long)e * g.rows + r) * wpr;
    const int ks = k0 + 8 * (j & 1);
    uint32_t v = 0;
    for (int q2 = 0; q2 < 8; ++q2) {
      const uint32_t code = get_code(g.fmt, row, ks + q2);
      const int n = tiled_nib(q2);
      v |= (code & 15u) << (4 * n);
      HW[j] |= (code >> 4) << (4 * n);
      P5 |= ((code >> 4) & 1u) << plane5_pos(j, n);
      P6[j >> 1] |= ((code >> 4) & 3u) << plane6_pos(j, n);
    }
    W[j] = v;
  }
  uint8_t* blkp = out + tiled_item(g, e, blk, c) + (long long)(w * g.ng + G) * tiled_cb(g.fmt);
  uint32_t* pl = reinterpret_cast<uint32_t*>(blkp) + lane;
  const int bits = tiled_bits(g.fmt);
  if (bits == 2 || bits == 3) {
    pl[0] = planes_l(W[0], W[1]);
    pl[32] = planes_l(W[2], W[3]);
    if (bits == 3) pl[64] = planes_h(W[0], W[1], W[2], W[3]);
  } else {
    *reinterpret_cast<uint4*>(blkp + lane * 16) = make_uint4(W[0], W[1], W[2], W[3]);
    uint32_t* hp = reinterpret_cast<uint32_t*>(blkp + 512) + lane;
    if (bits == 5) hp[0] = P5;
    if (bits == 6) {
      hp[0] = P6[0];
      hp[32] = P6[1];
    }
    if (bits == 8)
      *reinterpret_cast<uint4*>(blkp + 512 + lane * 16) = make_uint4(HW[0], HW[1], HW[2], HW[3]);
  }
}

// Scale-group size of a format and the number of its groups in one item.
__host__ __device__ inline int tiled_gsz(const TileGeo& g) {
  return g.fmt == MOE_FMT_W4A16_SYM_G128 ? 128 : 64;
}

// one thread per (expert, item, tile w, scale group G', fragment row g)
__global__ void k_repack_scales(TileGeo g, int E, const uint16_t* __restrict__ s,
                                const uint16_t* __restrict__ b, uint8_t* __restrict__ out) {
  const int gsz = tiled_gsz(g);
  const int nsg = g.CK / gsz;
  const long long n = (long long)E * g.nblk * g.nch * 8 * nsg * 8;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  long long q = i;
  const int gq = int(q % 8); q /= 8;
  const int G = int(q % nsg); q /= nsg;
  const int w = int(q % 8); q /= 8;
  const int c = int(q % g.nch); q /= g.nch;
  const int blk = int(q % g.nblk); q /= g.nblk;
  const int e = int(q);
  const int r0 = tiled_row(g, blk, w) + gq;
  const int gpr = g.K / gsz;
  const long long i0 = ((long long)e * g.rows + r0) * gpr + c * nsg + G;
  const long long i1 = i0 + 8LL * gpr;
  uint8_t* sc = out + tiled_item(g, e, blk, c) + g.code_bytes;
  if (g.fmt == MOE_FMT_W4A16_SYM_G128) {
    *reinterpret_cast<uint32_t*>(sc + ((w * 8 + gq) * nsg + G) * 4) =
        uint32_t(s[i0]) | (uint32_t(s[i1]) << 16);
  } else {
    *reinterpret_cast<uint2*>(sc + ((w * 8 + gq) * nsg + G) * 8) =
        make_uint2(uint32_t(s[i0]) | (uint32_t(b[i0]) << 16),
                   uint32_t(s[i1]) | (uint32_t(b[i1]) << 16));
  }
}

__device__ __forceinline__ uint32_t tiled_code(const TileGeo& g, const uint8_t* tl, int e, int r,
                                               int k) {
  const TiledPos p = tiled_pos(g, e, r, k);
  const int bits = tiled_bits(g.fmt);
  const uint32_t* pl = reinterpret_cast<const uint32_t*>(tl + p.block) + p.lane;
  if (bits == 2 || bits == 3) {
    uint32_t w0, w1, w2, w3;
    planes_to_words(pl[0], pl[32], bits == 3 ? pl[64] : 0u, w0, w1, w2, w3);
    const uint32_t W = p.widx == 0 ? w0 : p.widx == 1 ? w1 : p.widx == 2 ? w2 : w3;
    return (W >> (4 * p.nib)) & 15u;
  }
  const uint32_t lo =
      (reinterpret_cast<const uint32_t*>(tl + p.block + p.lane * 16)[p.widx] >> (4 * p.nib)) & 15u;
  const uint32_t* hp = reinterpret_cast<const uint32_t*>(tl + p.block + 512) + p.lane;
  uint32_t hi = 0;
  if (bits == 5) hi = (hp[0] >> plane5_pos(p.widx, p.nib)) & 1u;
  if (bits == 6) hi = (hp[32 * (p.widx >> 1)] >> plane6_pos(p.widx, p.nib)) & 3u;
  if (bits == 8)
    hi = (reinterpret_cast<const uint32_t*>(tl + p.block + 512 + p.lane * 16)[p.widx] >>
          (4 * p.nib)) & 15u;
  return lo | (hi << 4);
}

// one thread per canonical packed word
__global__ void k_unrepack_codes(TileGeo g, int E, const uint8_t* __restrict__ tl,
                                 uint32_t* __restrict__ wc) {
  const int bits = fmt_bits(g.fmt);
  const long wpr = long(g.K) * bits / 32;
  const long long n = (long long)E * g.rows * wpr;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const long long er = i / wpr;
  const int j = int(i - er * wpr);
  const int e = int(er / g.rows), r = int(er % g.rows);
  uint32_t v = 0;
  if (fmt_stream(g.fmt)) {
    for (int b = 0; b < 32; ++b) {
      const long s = long(j) * 32 + b;
      v |= ((tiled_code(g, tl, e, r, int(s / bits)) >> (s % bits)) & 1u) << b;
    }
  } else {
    const int per = 32 / bits;
    for (int q = 0; q < per; ++q) v |= tiled_code(g, tl, e, r, per * j + q) << (bits * q);
  }
  wc[i] = v;
}

// one thread per canonical scale (and bias) entry
__global__ void k_unrepack_scales(TileGeo g, int E, const uint8_t* __restrict__ tl,
                                  uint16_t* __restrict__ s, uint16_t* __restrict__ b) {
  const int gsz = tiled_gsz(g);
  const int gpr = g.K / gsz, nsg = g.CK / gsz;
  const long long n = (long long)E * g.rows * gpr;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const long long er = i / gpr;
  const int gi = int(i - er * gpr);
  const int e = int(er / g.rows), r = int(er % g.rows);
  int blk, w, sub;
  tiled_rowpos(g, r, blk, w, sub);
  const int c = gi / nsg, G = gi % nsg, gq = sub & 7, hi = sub >> 3;
  const uint8_t* sc = tl + tiled_item(g, e, blk, c) + g.code_bytes;
  if (g.fmt == MOE_FMT_W4A16_SYM_G128) {
    s[i] = reinterpret_cast<const uint16_t*>(sc + ((w * 8 + gq) * nsg + G) * 4)[hi];
  } else {
    const uint16_t* ent = reinterpret_cast<const uint16_t*>(sc + ((w * 8 + gq) * nsg + G) * 8);
    s[i] = ent[2 * hi];
    b[i] = ent[2 * hi + 1];
  }
}

unsigned blocks_for(long long n) { return unsigned((n + 255) / 256); }

}  // namespace

cudaError_t launch_repack(const TileGeo& g, int E, const uint32_t* wc, const uint16_t* s,
                          const uint16_t* b, uint8_t* tiled, cudaStream_t st) {
  const long long nc = (long long)E * g.nblk * g.nch * 8 * g.ng * 32;
  const long long ns = (long long)E * g.nblk * g.nch * 8 * (g.CK / tiled_gsz(g)) * 8;
  if (nc == 0) return cudaSuccess;
  k_repack_codes<<<blocks_for(nc), 256, 0, st>>>(g, E, wc, tiled);
  k_repack_scales<<<blocks_for(ns), 256, 0, st>>>(g, E, s, b, tiled);
  return cudaGetLastError();
}

cudaError_t launch_unrepack(const TileGeo& g, int E, const uint8_t* tiled, uint32_t* wc,
                            uint16_t* s, uint16_t* b, cudaStream_t st) {
  const long long nc = (long long)E * g.rows * (long long)g.K * fmt_bits(g.fmt) / 32;
  const long long ns = (long long)E * g.rows * (g.K / tiled_gsz(g));
  if (nc == 0) return cudaSuccess;
  k_unrepack_codes<<<blocks_for(nc), 256, 0, st>>>(g, E, tiled, wc);
  k_unrepack_scales<<<blocks_for(ns), 256, 0, st>>>(g, E, tiled, s, b);
  return cudaGetLastError();
}

cudaError_t launch_pack(int fmt, const uint8_t* codes, int rows, int cols, uint32_t* packed,
                        cudaStream_t st) {
  const long n = long(rows) * cols * fmt_bits(fmt) / 32;
  if (n == 0) return cudaSuccess;
  k_pack<<<unsigned((n + 255) / 256), 256, 0, st>>>(fmt, codes, rows, cols, packed);
  return cudaGetLastError();
}

cudaError_t launch_unpack(int fmt, const uint32_t* packed, int rows, int cols, uint8_t* codes,
                          cudaStream_t st) {
  const long n = long(rows) * cols;
  if (n == 0) return cudaSuccess;
  k_unpack<<<unsigned((n + 255) / 256), 256, 0, st>>>(fmt, packed, rows, cols, codes);
  return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, const void* q, const uint16_t* s, const uint16_t* b, int rows,
                           int cols, float* w, cudaStream_t st) {
  const long n = long(rows) * cols;
  if (n == 0) return cudaSuccess;
  k_dequant<<<unsigned((n + 255) / 256), 256, 0, st>>>(fmt, q, s, b, rows, cols, w);
  return cudaGetLastError();
}

}  // namespace moe
