// prefill.h -- the prefill expert GEMMs on the 5th-generation tensor cores.
#pragma once

#include "kernels.h"

namespace moe {

constexpr int kPfTile = 128;   // tokens per N tile (tensor-memory columns per accumulator)
constexpr int kPfThreads = 576;
// Experts with at most this many assignments in a prefill call go to the
// decode units instead (each tensor-core unit dequantises a whole weight
// block whatever its rows; the decode units cost per 8 rows).
constexpr int kPfLight = 16;

// One prefill GEMM launch over a tile list: each tile is <= kPfTile rows of
// one expert; every (tile, 128-row weight block) is a unit.
//   mode 0 (gate/up): A = w13 blocks (64 gate + 64 up rows), B = fp16
//     activation rows, epilogue h = silu(gate) * up -> fp16 h rows off + n;
//   mode 1 (down): A = w2 blocks (128 rows), B = fp16 h rows off + n,
//     epilogue fp32 y rows (scattered by perm, or off + n).
// The dequantised weights enter the MMA as fp16, fma(s, q, b) rounded once;
// accumulation is fp32.
struct PrefillJob {
  TileGeo g;                 // tiled geometry of the matrix
  const uint8_t* base;       // tiled bank (expert 0, item 0)
  const int* n_tiles;        // device tile count, or nullptr: fixed tiles over fixed_T rows
  const int* te;             // tile -> expert
  const int* toff;           //         first bucket position (or row)
  const int* tcnt;           //         rows (1..kPfTile)
  int fixed_e, fixed_T;
  int max_tiles;             // host bound (unused by the kernel)
  const uint16_t* B;         // fp16 operand rows (x, or h), ldB elements apart
  int ldB;
  int gather;                // mode 0: operand row = perm[off + n] / k (else off + n)
  const int* perm;
  int k;
  uint16_t* h;               // mode 0 output: fp16 h, ldh elements apart
  int ldh;
  float* y;                  // mode 1 output (fp32), ldy elements apart
  int ldy;
  int scatter;               // mode 1: output row = perm[off + n] (else off + n)
  int* status;
  // Optional second bank of the same geometry (the shared expert, expert 0
  // of sh_base) run in the same launch: its units come first, fixed tiles
  // over sh_T rows, operand rows sh_B + row * ldB (never gathered), outputs
  // sh_h (mode 0, ldh) or sh_y (mode 1, ldy; never scattered).
  const uint8_t* sh_base;    // nullptr: none
  int sh_T;
  const uint16_t* sh_B;
  uint16_t* sh_h;
  float* sh_y;
};

// Shared memory of a launch for geometry g in mode 0/1 (0: not supported).
int prefill_smem(const TileGeo& g, int mode);
cudaError_t launch_prefill(const PrefillJob& J, int mode, int sms, cudaStream_t st);
// bf16 activations [n] -> fp16 (exact in fp16's normal range; outside it the
// status word gets MOE_ERR_RANGE); n a multiple of 8, both 16-byte aligned
cudaError_t launch_act_f16(const uint16_t* x, long n, uint16_t* xh, int* status,
                           cudaStream_t st);

}  // namespace moe
