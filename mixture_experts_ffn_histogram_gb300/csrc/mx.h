// Internal launchers of the MXFP8 forward path (host side).  Arguments were
// validated by the C entry points in api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Geometry of the MX operands (see include/moe.h for the layouts).
constexpr int kMxBlock = 32;      // elements sharing one scale
constexpr int kMxKBlock = 128;    // elements of one k-block (one 512-byte scale block)
constexpr int kMxRowsPerTile = 128;

inline long mx_cdiv(long a, long b) { return (a + b - 1) / b; }
// k-blocks of a contraction of length k
inline long mx_kblocks(long k) { return mx_cdiv(k, kMxKBlock); }
// upper bound on the 128-row tiles of all groups together: sum over groups
// of ceil(rows/128) <= ceil(R/128) + E
inline long mx_tile_bound(const moe_dims& d) {
  return mx_cdiv(static_cast<long>(d.T) * d.K, kMxRowsPerTile) + d.E;
}
// 128-row blocks of a weight's output rows, rounded up to whole 256-row tiles
inline long mx_weight_row_blocks(long n) { return 2 * mx_cdiv(n, 256); }
// token-axis (transposed) operands: each group padded to whole 128-row tiles,
// the tiles numbered as in the tile-blocked scales
inline long mx_token_cols(const moe_dims& d) { return kMxRowsPerTile * mx_tile_bound(d); }

// w [E][Kd][N] quantized along Kd into the transposed weight layout (codes
// [E][N][Kd], FC1 rows interleaved when fc1_interleave) and/or along N in
// its own layout (q2, sc2: codes [E][Kd][N], scales [E][KB(N)][NBp(Kd)][512]);
// either pair may be null, one read of w serves both.
cudaError_t launch_mx_quantize_weights(const uint16_t* w, uint8_t* q, uint8_t* sc, uint8_t* q2,
                                       uint8_t* sc2, int E, int Kd, int N, bool fc1_interleave,
                                       cudaStream_t s);
cudaError_t launch_mx_permute_quantize(const uint16_t* x, const int32_t* pos, const int32_t* offs,
                                       uint8_t* xq, uint8_t* xsc, const moe_dims& d,
                                       cudaStream_t s);

// Token-axis quantization: src [R, C] in expert-sorted order, or (row_src
// given) x [T, C] read at token row_src[r] / K -> codes [C, Rp] and scales
// [TB, NBp(C), 512] (TB tiles, Rp = 128 * TB; each group's rows padded with
// zeros to whole 128-row tiles).
cudaError_t launch_mx_quantize_tokens(const uint16_t* src, const int32_t* row_src,
                                      const int32_t* offs, uint8_t* qt, uint8_t* sct, int C,
                                      const moe_dims& d, cudaStream_t s);
// Row quantization of an expert-sorted [R, C] (blocks along C, tile-blocked scales).
cudaError_t launch_mx_quantize_rows(const uint16_t* src, const int32_t* offs, uint8_t* q,
                                    uint8_t* sc, int C, const moe_dims& d, cudaStream_t s);
enum class MxKind : int {
  kFc1 = 0,            // FC1 + SwiGLU: h (MX and/or bf16), optionally z
  kRows = 1,           // out[r, n] = sum_k A[r, k] * B_e[n, k], bf16
  kRowsSwigluBwd = 2,  // kRows with N = F, then dz = SwiGLU backward at z
  kWgrad = 3           // out[e, m, n] = sum over group e's tokens of A[m, t] * B[n, t]
};

struct MxGemmCall {
  MxKind kind;
  const uint8_t* a;         // row-quantized activations, or (kWgrad) token-axis codes [M, Rp]
  const uint8_t* a_sc;      // their scales
  const uint8_t* b;         // the quantized weight, or (kWgrad) token-axis codes [N, Rp]
  const uint8_t* b_sc;      // its scales
  const int32_t* offs;      // group offsets [E+1]
  uint8_t* hq;              // kFc1: h codes, or nullptr
  uint8_t* hsc;             // kFc1: h scales, or nullptr
  uint16_t* out;            // kFc1: h bf16 or nullptr; kRows: [R, n]; kRowsSwigluBwd: dz
                            // [R, 2F]; kWgrad: [E, m, n]
  const uint16_t* z_in;     // kRowsSwigluBwd: z [R, 2F]
  uint16_t* z_out;          // kFc1: z [R, 2F] or nullptr
  int32_t* dev_status;
  moe_dims d;
  int kd;                   // kRows: contraction length
  int n;                    // kRows, kWgrad: output columns (B rows per expert)
  int m;                    // kWgrad: output rows per expert (A rows)
};
cudaError_t launch_mx_grouped_gemm(const MxGemmCall& c, cudaStream_t s);

}  // namespace moe
