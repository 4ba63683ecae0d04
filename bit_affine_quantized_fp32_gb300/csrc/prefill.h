// prefill.h -- the prefill expert GEMMs on the 5th-generation tensor cores.
#pragma once

#include "kernels.h"

namespace moe {

constexpr int kPfTile = 128;   // tokens per N tile (tensor-memory columns per accumulator)
constexpr int kPfThreads = 480;
// Experts with at most this many assignments in a prefill call go to the
// decode units instead (each tensor-core unit dequantises a whole weight
// block whatever its rows; the decode units cost per 8 rows).
constexpr int kPfLight = 40;

// One prefill GEMM launch over a tile list: each tile is <= kPfTile rows of
// one expert; every (tile, 128-row weight block) is a unit.
//   mode 0 (gate/up): A = w13 blocks (64 gate + 64 up rows), B = activation
//     rows, epilogue h = silu(gate) * up -> h rows off + n as bf16 hi + lo;
//   mode 1 (down): A = w2 blocks (128 rows), B = h rows off + n (hi + lo),
//     epilogue fp32 y rows (scattered by perm, or off + n).
// The dequantised weights enter the MMA as bf16 hi + lo parts as well (fp16
// for fp16 activations), so products carry ~16 significant bits and the sums
// fp32 rounding only.
struct PrefillJob {
  TileGeo g;                 // tiled geometry of the matrix
  const uint8_t* base;       // tiled bank (expert 0, item 0)
  const int* n_tiles;        // device tile count, or nullptr: fixed tiles over fixed_T rows
  const int* te;             // tile -> expert
  const int* toff;           //         first bucket position (or row)
  const int* tcnt;           //         rows (1..kPfTile)
  int fixed_e, fixed_T;
  int max_tiles;             // host bound (unused by the kernel)
  const uint16_t* B;         // operand rows (x, or h hi), ldB elements apart
  const uint16_t* Blo;       // mode 1: h lo rows
  int ldB;
  int gather;                // mode 0: operand row = perm[off + n] / k (else off + n)
  const int* perm;
  int k;
  uint16_t* h;               // mode 0 output: bf16 h hi, ldh elements apart
  uint16_t* hl;              //                bf16 h lo (h - hi)
  int ldh;
  float* y;                  // mode 1 output (fp32), ldy elements apart
  int ldy;
  size_t yzero;              // mode 1: when > 0, 0 is also stored at y[i + yzero] (the
                             //         second k-half plane the decode units would write)
  int scatter;               // mode 1: output row = perm[off + n] (else off + n)
  int* status;
};

// Shared memory of a launch for geometry g in mode 0/1 (0: not supported).
int prefill_smem(const TileGeo& g, int mode);
// mode 0/1 as above; f16a: fp16 activations (mode 0 only).
cudaError_t launch_prefill(const PrefillJob& J, int mode, bool f16a, int sms, cudaStream_t st);

}  // namespace moe
