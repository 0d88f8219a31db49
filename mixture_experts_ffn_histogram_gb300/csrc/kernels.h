// Internal launchers of libmoe.so (host side).  Each returns the status of
// its launches; arguments were validated by the C entry points in api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Routing scratch (a caller workspace, or the no-allocation call's fixed
// array): the grid barrier's word inside the first kRouteBarrierBytes, then
// one int32 per (block, expert) for the blocks' per-expert totals, for up to
// `max_blocks` blocks.  A block of the routing kernel covers at least one
// token and there is at most one block per SM, so min(T, kRouteBlocksBound)
// blocks bound the grid on any device.
constexpr size_t kRouteBarrierBytes = 256;
constexpr long kRouteBlocksBound = 1024;
inline long route_max_blocks(int T) { return T < kRouteBlocksBound ? T : kRouteBlocksBound; }
inline size_t route_ws_bytes(const moe_dims& d) {
  return kRouteBarrierBytes + static_cast<size_t>(route_max_blocks(d.T)) *
                                  static_cast<size_t>(d.E) * sizeof(int32_t);
}

// Routing over `max_blocks` blocks at most (the per-block totals that fit in
// `scratch` after the barrier word).
cudaError_t launch_route_histogram(const float* logits, const float* bias, int mode, int32_t* ids,
                                   float* w, int32_t* group_sizes, int32_t* group_offsets,
                                   int32_t* pos, int32_t* row_src, int32_t* dev_status,
                                   void* scratch, long max_blocks, const moe_dims& d,
                                   cudaStream_t s);

// Capacity, in int32, of the fixed scratch of the no-allocation routing
// call.  Its documented limit, 2 * ceil(T/256) * E <= this, is what the C
// entry point checks; the kernel needs less.
constexpr size_t kRouteStaticScratchInts = 262144;  // 1 MiB
inline int route_chunks(int T) { return (T + 255) / 256; }
cudaError_t launch_route_histogram_static(const float* logits, const float* bias, int mode,
                                          int32_t* ids, float* w, int32_t* group_sizes,
                                          int32_t* group_offsets, int32_t* pos, int32_t* row_src,
                                          int32_t* dev_status, const moe_dims& d, cudaStream_t s);

cudaError_t launch_permute(const uint16_t* x, const int32_t* pos, uint16_t* xs, const moe_dims& d,
                           cudaStream_t s);
cudaError_t launch_combine(const uint16_t* ys, const float* w, const int32_t* pos, uint16_t* out,
                           const moe_dims& d, cudaStream_t s);
cudaError_t launch_combine_bwd(const uint16_t* dout, const uint16_t* ys, const float* w,
                               const int32_t* pos, uint16_t* dys, float* dw, const moe_dims& d,
                               cudaStream_t s);
// the combine backward that also writes dys quantized along D (MXFP8 codes
// [R][D] and tile-blocked scales of the rows' groups)
cudaError_t launch_mx_combine_bwd(const uint16_t* dout, const uint16_t* ys, const float* w,
                                  const int32_t* pos, const int32_t* offs, uint16_t* dys,
                                  uint8_t* dyq, uint8_t* dysc, float* dw, const moe_dims& d,
                                  cudaStream_t s);
cudaError_t launch_swiglu_bwd(const uint16_t* dh, const uint16_t* z, uint16_t* dz, long R, int F,
                              cudaStream_t s);
cudaError_t launch_bounded_wait_selftest(int32_t* dev_status, uint64_t limit_ns, cudaStream_t s);
// out = bf16(acc) elementwise, n elements (a multiple of 8)
cudaError_t launch_acc_to_bf16(const float* acc, uint16_t* out, long n, cudaStream_t s);

// Grouped GEMMs (tcgen05).  `rows` = T*K.
// kFc1Gather: FC1 whose rows are gathered from the token-major x by row_src
// (no permuted copy); kFc2Combine: FC2 whose rows are weighted by w and added
// into an fp32 [T, D] accumulator (no ys, no separate combine).
enum class GemmKind : int {
  kFc1 = 0, kFc2 = 1, kDlhsFc2 = 2, kDlhsFc1 = 3, kDrhsFc2 = 4, kDrhsFc1 = 5,
  kFc1Gather = 6, kFc2Combine = 7
};

struct GemmCall {
  GemmKind kind;
  const void* a;           // left operand base (xs, h, dys, dz, or h/xs for drhs)
  const void* b;           // right operand base (wi, wo, or dys/dz for drhs)
  const int32_t* offs;     // group offsets [E+1]
  void* out0;              // h / ys / dz-or-dh / dxs / dwo / dwi
  void* out1;              // z (FC1) or nullptr
  const void* aux;         // z for the fused SwiGLU backward, or nullptr
  int32_t* dev_status;
  moe_dims d;
  unsigned int* tile_ctr = nullptr;  // drhs: a device counter for the dynamic tile schedule
  const int32_t* row_src = nullptr;  // gather / combine: slot j = t*K + k of each sorted row
  const float* w = nullptr;          // combine: routing weights [T, K]
  float* acc = nullptr;              // combine: fp32 [T, D] accumulator
};

// Bytes at the start of `ws` that hold the drhs tile counter; the SwiGLU
// backward's dz scratch follows them.
constexpr size_t kWsCounterBytes = 256;

cudaError_t launch_grouped_gemm(const GemmCall& c, cudaStream_t s);

int sm_count();

}  // namespace moe
