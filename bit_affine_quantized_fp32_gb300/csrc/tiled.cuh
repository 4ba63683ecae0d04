// tiled.cuh -- geometry of the kernel-tiled expert layout.
//
// An expert's w13 (gate rows 0..I-1, up rows I..2I-1 of [2I, H]) and w2
// ([H, I]) are cut into items:
//   block   w13: 64 gate rows 64j.. + the 64 matching up rows I+64j..;
//           w2 : 128 rows 128r..;  eight 16-row M-tiles per block, tile w;
//   chunk   CK consecutive reduction columns (512, else 256, else 128),
//           ng = CK/64 code groups;
//   item    (block, chunk) = [codes][scales] contiguous, items ordered
//           (block, chunk) inside an expert, experts one after another.
// Codes of an item, in MMA fragment order: for tile w, group G and lane
// (g = lane/4, t = lane%4), with rows r0 = tile row + g and r1 = r0 + 8 and
// codes k0 = c*CK + 64G + 16t, the four 8-code words
//   W0 = codes r0[k0, k0+8)   W1 = codes r0[k0+8, k0+16)
//   W2 = codes r1[k0, k0+8)   W3 = codes r1[k0+8, k0+16)
// where code j (0..7) of a word sits in nibble (j&1)*4 + j/2, i.e. the
// nibbles hold codes [0 2 4 6 1 3 5 7]: nibbles i and i+4 are the adjacent
// pair (2i, 2i+1), which is how an MMA register takes two k-values, so the
// activations stay in their natural order.
// A (w, G) code block holds exactly the codes' bits (128 * bits bytes), the
// words W0..W3 above holding each code's low 4 bits:
//   4-bit / W4A16: 16 bytes [W0 W1 W2 W3] per lane, blocks of 512 B.
//   3-bit: three 32-bit planes per block of 384 B, plane p holding lane l's
//     word at p*128 + 4l:
//       L01 = (W0 & 0x33333333) | (W1 & 0x33333333) << 2      (bits 0-1)
//       L23 = (W2 & 0x33333333) | (W3 & 0x33333333) << 2
//       H   = (W0 >> 2 & 0x11111111) | (W1 >> 1 & 0x22222222)
//           | (W2 & 0x44444444) | (W3 << 1 & 0x88888888)        (bit 2)
//   2-bit: the planes L01 and L23 alone (256 B).
//   5-bit: [W0..W3] per lane (512 B), then a plane (128 B) of bit 4: bit 4 of
//     the code in nibble n of Wx sits at bit 4x + (n & 3) + 16 (n >> 2), so
//     (plane >> (4x + m - 4)) puts the bits of the code pair in nibbles m and
//     m + 4 at bits 4 and 20, next to the low nibbles.
//   6-bit: [W0..W3] (512 B), then two planes (bits 4-5 of the codes of W0,W1
//     and of W2,W3): bits 4-5 of the code in nibble n of Wx at bit
//     2 (4 (x & 1) + (n & 3)) + 16 (n >> 2) of plane x >> 1.
//   8-bit: [W0..W3] of the low nibbles, then the same 16 bytes per lane of
//     the high nibbles (1024 B).
// Scales of an item (fp16), one run per (w, g) so that a lane's groups are
// contiguous:
//   affine: entry (w, g, G) = [s(r0), b(r0), s(r1), b(r1)] of 64-group G,
//           8 bytes at ((w*8 + g)*ng + G)*8;
//   W4A16 : entry (w, g, G') = [s(r0), s(r1)] of 128-group G', 4 bytes at
//           ((w*8 + g)*(ng/2) + G')*4.
#pragma once

#include "common.cuh"

namespace moe {

struct TileGeo {
  int fmt;
  int down;         // 0: w13, 1: w2
  int inter;        // I
  int rows;         // 2I or H
  int K;            // H or I
  int CK;           // chunk
  int nch;          // K / CK
  int ng;           // CK / 64
  int nblk;         // blocks per expert
  int code_bytes;   // per item
  int sc_bytes;     // per item
  int item_bytes;   // code_bytes + sc_bytes
  long long expert_bytes;
};

// bits per code of an expert format
__host__ __device__ constexpr int tiled_bits(int fmt) {
  return fmt == MOE_FMT_AFFINE2_G64   ? 2
         : fmt == MOE_FMT_AFFINE3_G64 ? 3
         : fmt == MOE_FMT_AFFINE5_G64 ? 5
         : fmt == MOE_FMT_AFFINE6_G64 ? 6
         : fmt == MOE_FMT_AFFINE8_G64 ? 8
                                      : 4;
}
// bytes of one (w, G) code block
__host__ __device__ constexpr int tiled_cb(int fmt) { return 128 * tiled_bits(fmt); }

__host__ __device__ inline int tiled_chunk(int K) {
  return K % 512 == 0 ? 512 : (K % 256 == 0 ? 256 : 128);
}

__host__ __device__ inline TileGeo tile_geo(int fmt, int inter, int hidden, int down) {
  TileGeo g;
  g.fmt = fmt;
  g.down = down;
  g.inter = inter;
  g.rows = down ? hidden : 2 * inter;
  g.K = down ? inter : hidden;
  g.CK = tiled_chunk(g.K);
  g.nch = g.K / g.CK;
  g.ng = g.CK / 64;
  g.nblk = down ? hidden / 128 : inter / 64;
  g.code_bytes = 8 * g.ng * tiled_cb(fmt);
  g.sc_bytes = fmt == MOE_FMT_W4A16_SYM_G128 ? 8 * (g.ng / 2) * 8 * 4 : 8 * g.ng * 8 * 8;
  g.item_bytes = g.code_bytes + g.sc_bytes;
  g.expert_bytes = (long long)g.nblk * g.nch * g.item_bytes;
  return g;
}

// Nibble of code j (0..7) inside its tiled word.
__host__ __device__ inline int tiled_nib(int j) { return (j & 1) * 4 + (j >> 1); }

// First matrix row of M-tile w of block blk.
__host__ __device__ inline int tiled_row(const TileGeo& g, int blk, int w) {
  if (g.down) return blk * 128 + 16 * w;
  return w < 4 ? blk * 64 + 16 * w : g.inter + blk * 64 + 16 * (w - 4);
}

__host__ __device__ inline uint32_t planes_l(uint32_t wa, uint32_t wb) {
  return (wa & 0x33333333u) | ((wb & 0x33333333u) << 2);
}

__host__ __device__ inline uint32_t planes_h(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
  return ((w0 >> 2) & 0x11111111u) | ((w1 >> 1) & 0x22222222u) | (w2 & 0x44444444u) |
         ((w3 << 1) & 0x88888888u);
}

// Bit position, in a 5-bit block's bit-4 plane, of the code in nibble n of
// word x; in a 6-bit block's plane x >> 1, of bit 4 of that code (bit 5 next).
__host__ __device__ inline int plane5_pos(int x, int n) { return 4 * x + (n & 3) + 16 * (n >> 2); }
__host__ __device__ inline int plane6_pos(int x, int n) {
  return 2 * (4 * (x & 1) + (n & 3)) + 16 * (n >> 2);
}

// Inverse of the planes: the four 8-code words of a 3-bit fragment.
__device__ __forceinline__ void planes_to_words(uint32_t l01, uint32_t l23, uint32_t h,
                                                uint32_t& w0, uint32_t& w1, uint32_t& w2,
                                                uint32_t& w3) {
  w0 = (l01 & 0x33333333u) | ((h << 2) & 0x44444444u);
  w1 = ((l01 >> 2) & 0x33333333u) | ((h << 1) & 0x44444444u);
  w2 = (l23 & 0x33333333u) | (h & 0x44444444u);
  w3 = ((l23 >> 2) & 0x33333333u) | ((h >> 1) & 0x44444444u);
}

}  // namespace moe
