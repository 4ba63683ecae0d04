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

namespace moe {

namespace {

__host__ __device__ inline int fmt_bits(int fmt) {
  switch (fmt) {
    case MOE_FMT_AFFINE8_G64: return 8;
    case MOE_FMT_AFFINE4_G64: return 4;
    case MOE_FMT_AFFINE3_G64: return 3;
    case MOE_FMT_W4A16_SYM_G128: return 4;
    default: return 0;
  }
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
  if (fmt == MOE_FMT_AFFINE3_G64) {
    for (int b = 0; b < 32; ++b) {
      const long s = j * 32 + b;
      const uint32_t code = row[s / 3];
      v |= ((code >> (s % 3)) & 1u) << b;
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
  if (fmt == MOE_FMT_AFFINE3_G64) {
    const long s = 3 * c;
    const long w = s >> 5;
    const int b = int(s & 31);
    uint32_t v = row[w] >> b;
    if (b > 29) v |= row[w + 1] << (32 - b);
    return v & 7u;
  }
  const int bits = fmt_bits(fmt);
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

}  // namespace

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
