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

cudaError_t launch_mx_quantize_weights(const uint16_t* w, uint8_t* q, uint8_t* sc, int E, int Kd,
                                       int N, bool fc1_interleave, cudaStream_t s);
cudaError_t launch_mx_permute_quantize(const uint16_t* x, const int32_t* pos, const int32_t* offs,
                                       uint8_t* xq, uint8_t* xsc, const moe_dims& d,
                                       cudaStream_t s);

struct MxGemmCall {
  bool fc1;                 // FC1 + SwiGLU (else FC2)
  const uint8_t* a;         // xq or hq
  const uint8_t* a_sc;      // their tile-blocked scales
  const uint8_t* b;         // the quantized weight
  const uint8_t* b_sc;      // its blocked scales
  const int32_t* offs;      // group offsets [E+1]
  uint8_t* hq;              // FC1: h codes, or nullptr
  uint8_t* hsc;             // FC1: h scales, or nullptr
  uint16_t* out;            // FC1: h bf16 or nullptr; FC2: ys
  int32_t* dev_status;
  moe_dims d;
};
cudaError_t launch_mx_grouped_gemm(const MxGemmCall& c, cudaStream_t s);

}  // namespace moe
