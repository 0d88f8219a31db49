// C entry points of libmoe.so: argument checks, workspace carving, launches.
// The operations and their sources are documented in include/moe.h.
#include <atomic>
#include <cstdint>

#include "kernels.h"
#include "moe.h"
#include "mx.h"

namespace moe {

int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) dev = 0;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    v = 148;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

}  // namespace moe

namespace {

using moe::GemmCall;
using moe::GemmKind;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

moe_status check_dims(const moe_dims& d) {
  if (d.T < 0 || d.D <= 0 || d.F <= 0 || d.E <= 0 || d.K <= 0) return MOE_ERR_UNSUPPORTED;
  if (d.D % 64 != 0 || d.F % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (d.K > d.E || d.K > 32 || d.E > 1024) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d.T) * d.K >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int64_t rows(const moe_dims& d) { return static_cast<int64_t>(d.T) * d.K; }

size_t dz_ws_bytes(const moe_dims& d) {
  return static_cast<size_t>(rows(d)) * 2u * static_cast<size_t>(d.F) * 2u;
}

}  // namespace

#define MOE_CHECK_DIMS(d)                          \
  do {                                             \
    moe_status st_ = check_dims(d);                \
    if (st_ != MOE_OK) return st_;                 \
  } while (0)
#define MOE_REQUIRE(p)                             \
  do {                                             \
    if (!ok_ptr(p)) return MOE_ERR_INVALID_ARG;    \
  } while (0)
#define MOE_OPTIONAL(p)                                        \
  do {                                                         \
    if ((p) != nullptr && !aligned16(p)) return MOE_ERR_INVALID_ARG; \
  } while (0)

extern "C" {

size_t moe_workspace_bytes(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  size_t need = moe::route_ws_bytes(d);
  const size_t dz = moe::kWsCounterBytes + dz_ws_bytes(d);
  if (dz > need) need = dz;
  return (need + 255u) & ~static_cast<size_t>(255u);
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer)";
    case MOE_ERR_UNSUPPORTED: return "unsupported dimensions";
    case MOE_ERR_CUDA: return "CUDA launch error";
    case MOE_ERR_DEVICE: return "expert id outside [0, E) seen on the device";
    case MOE_ERR_TIMEOUT: return "a bounded wait inside a kernel timed out";
  }
  return "unknown status";
}

int moe_abi_version(void) { return 4; }

moe_status moe_route_histogram(const float* logits, const float* bias, moe_score_mode mode,
                               int32_t* ids, float* w, int32_t* group_sizes,
                               int32_t* group_offsets, int32_t* pos, int32_t* row_src,
                               int32_t* dev_status, void* ws, moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (mode != MOE_SCORE_SOFTMAX_TOPK && mode != MOE_SCORE_SIGMOID_NORM && mode != MOE_SCORE_GIVEN)
    return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE(group_sizes);
  MOE_REQUIRE(group_offsets);
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(bias);
  if (d.T > 0) {
    MOE_REQUIRE(ids);
    MOE_REQUIRE(pos);
    MOE_REQUIRE(row_src);
    MOE_REQUIRE(ws);
    if (mode != MOE_SCORE_GIVEN) {
      MOE_REQUIRE(logits);
      MOE_REQUIRE(w);
    } else {
      MOE_OPTIONAL(w);
    }
  }
  return from_cuda(moe::launch_route_histogram(logits, bias, static_cast<int>(mode), ids, w,
                                               group_sizes, group_offsets, pos, row_src,
                                               dev_status, ws, moe::route_max_blocks(d.T), d,
                                               stream));
}

moe_status moe_route_histogram_noalloc(const float* logits, const float* bias, moe_score_mode mode,
                                       int32_t* ids, float* w, int32_t* group_sizes,
                                       int32_t* group_offsets, int32_t* pos, int32_t* row_src,
                                       int32_t* dev_status, moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (mode != MOE_SCORE_SOFTMAX_TOPK && mode != MOE_SCORE_SIGMOID_NORM && mode != MOE_SCORE_GIVEN)
    return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE(group_sizes);
  MOE_REQUIRE(group_offsets);
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(bias);
  if (d.T > 0) {
    MOE_REQUIRE(ids);
    MOE_REQUIRE(pos);
    MOE_REQUIRE(row_src);
    if (mode != MOE_SCORE_GIVEN) {
      MOE_REQUIRE(logits);
      MOE_REQUIRE(w);
    } else {
      MOE_OPTIONAL(w);
    }
  }
  const size_t need = 2u * static_cast<size_t>(moe::route_chunks(d.T)) * static_cast<size_t>(d.E);
  if (need > moe::kRouteStaticScratchInts) return MOE_ERR_UNSUPPORTED;
  return from_cuda(moe::launch_route_histogram_static(logits, bias, static_cast<int>(mode), ids, w,
                                                      group_sizes, group_offsets, pos, row_src,
                                                      dev_status, d, stream));
}

moe_status moe_permute(const moe_bf16* x, const int32_t* pos, moe_bf16* xs, moe_dims d,
                       cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(x);
  MOE_REQUIRE(pos);
  MOE_REQUIRE(xs);
  return from_cuda(moe::launch_permute(x, pos, xs, d, stream));
}

moe_status moe_permute_bwd(const moe_bf16* dxs, const int32_t* pos, moe_bf16* dx, moe_dims d,
                           cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(dxs);
  MOE_REQUIRE(pos);
  MOE_REQUIRE(dx);
  return from_cuda(moe::launch_combine(dxs, nullptr, pos, dx, d, stream));
}

moe_status moe_combine(const moe_bf16* ys, const float* w, const int32_t* pos, moe_bf16* out,
                       moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(ys);
  MOE_REQUIRE(w);
  MOE_REQUIRE(pos);
  MOE_REQUIRE(out);
  return from_cuda(moe::launch_combine(ys, w, pos, out, d, stream));
}

moe_status moe_fused_forward(const moe_bf16* x, const float* w, const int32_t* row_src,
                             const int32_t* group_offsets, const moe_bf16* wi, const moe_bf16* wo,
                             moe_bf16* h, float* acc, moe_bf16* out, int32_t* dev_status,
                             void* ws, moe_dims d, cudaStream_t stream) {
  (void)ws;
  MOE_CHECK_DIMS(d);
  MOE_OPTIONAL(dev_status);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(x);
  MOE_REQUIRE(w);
  MOE_REQUIRE(row_src);
  MOE_REQUIRE(group_offsets);
  MOE_REQUIRE(wi);
  MOE_REQUIRE(wo);
  MOE_REQUIRE(h);
  MOE_REQUIRE(acc);
  MOE_REQUIRE(out);
  GemmCall c1{GemmKind::kFc1Gather, x, wi, group_offsets, h, nullptr, nullptr, dev_status, d};
  c1.row_src = row_src;
  cudaError_t err = moe::launch_grouped_gemm(c1, stream);
  if (err != cudaSuccess) return from_cuda(err);
  const size_t n = static_cast<size_t>(d.T) * static_cast<size_t>(d.D);
  err = cudaMemsetAsync(acc, 0, n * sizeof(float), stream);
  if (err != cudaSuccess) return from_cuda(err);
  GemmCall c2{GemmKind::kFc2Combine, h, wo, group_offsets, nullptr, nullptr, nullptr, dev_status, d};
  c2.row_src = row_src;
  c2.w = w;
  c2.acc = acc;
  err = moe::launch_grouped_gemm(c2, stream);
  if (err != cudaSuccess) return from_cuda(err);
  return from_cuda(moe::launch_acc_to_bf16(acc, out, static_cast<long>(n), stream));
}

moe_status moe_combine_bwd(const moe_bf16* dout, const moe_bf16* ys, const float* w,
                           const int32_t* pos, moe_bf16* dys, float* dw, moe_dims d,
                           cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(dout);
  MOE_REQUIRE(ys);
  MOE_REQUIRE(w);
  MOE_REQUIRE(pos);
  MOE_REQUIRE(dys);
  MOE_REQUIRE(dw);
  return from_cuda(moe::launch_combine_bwd(dout, ys, w, pos, dys, dw, d, stream));
}

moe_status moe_grouped_gemm_fc1_swiglu(const moe_bf16* xs, const moe_bf16* wi,
                                       const int32_t* group_offsets, moe_bf16* h, moe_bf16* z,
                                       int32_t* dev_status, void* ws, moe_dims d,
                                       cudaStream_t stream) {
  (void)ws;
  MOE_CHECK_DIMS(d);
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(z);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(xs);
  MOE_REQUIRE(wi);
  MOE_REQUIRE(group_offsets);
  MOE_REQUIRE(h);
  GemmCall c{GemmKind::kFc1, xs, wi, group_offsets, h, z, nullptr, dev_status, d};
  return from_cuda(moe::launch_grouped_gemm(c, stream));
}

// Dims of a GEMM over experts [e_begin, e_end): the R = T*K rows are passed
// as T = R, K = 1 (the grouped GEMMs use only R), E = the range's experts.
static moe_dims range_dims(const moe_dims& d, int32_t e_begin, int32_t e_end) {
  moe_dims r = d;
  r.T = d.T * d.K;
  r.K = 1;
  r.E = e_end - e_begin;
  return r;
}

moe_status moe_grouped_gemm_fc1_swiglu_experts(const moe_bf16* xs, const moe_bf16* wi_part,
                                               const int32_t* group_offsets, int32_t e_begin,
                                               int32_t e_end, moe_bf16* h, moe_bf16* z,
                                               int32_t* dev_status, void* ws, moe_dims d,
                                               cudaStream_t stream) {
  (void)ws;
  MOE_CHECK_DIMS(d);
  if (e_begin < 0 || e_end <= e_begin || e_end > d.E) return MOE_ERR_INVALID_ARG;
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(z);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(xs);
  MOE_REQUIRE(wi_part);
  MOE_REQUIRE(group_offsets);  // the caller's whole array; the range reads a 4-byte-aligned slice
  MOE_REQUIRE(h);
  GemmCall c{GemmKind::kFc1, xs, wi_part, group_offsets + e_begin, h, z, nullptr, dev_status,
             range_dims(d, e_begin, e_end)};
  return from_cuda(moe::launch_grouped_gemm(c, stream));
}

moe_status moe_grouped_gemm_fc1_bwd_experts(const moe_bf16* dz, const moe_bf16* xs,
                                            const moe_bf16* wi_part,
                                            const int32_t* group_offsets, int32_t e_begin,
                                            int32_t e_end, moe_bf16* dxs, moe_bf16* dwi_part,
                                            int32_t* dev_status, void* ws, moe_dims d,
                                            cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (e_begin < 0 || e_end <= e_begin || e_end > d.E) return MOE_ERR_INVALID_ARG;
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(dxs);
  MOE_OPTIONAL(dwi_part);
  if (dxs == nullptr && dwi_part == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE(group_offsets);
  const moe_dims rd = range_dims(d, e_begin, e_end);
  const int32_t* offs = group_offsets + e_begin;
  if (d.T > 0) {
    MOE_REQUIRE(dz);
    if (dxs != nullptr) MOE_REQUIRE(wi_part);
    if (dwi_part != nullptr) {
      MOE_REQUIRE(xs);
      MOE_REQUIRE(ws);
    }
  }
  if (dxs != nullptr && d.T > 0) {
    GemmCall c{GemmKind::kDlhsFc1, dz, wi_part, offs, dxs, nullptr, nullptr, dev_status, rd};
    moe_status st = from_cuda(moe::launch_grouped_gemm(c, stream));
    if (st != MOE_OK) return st;
  }
  if (dwi_part != nullptr) {
    GemmCall c{GemmKind::kDrhsFc1, xs, dz, offs, dwi_part, nullptr, nullptr, dev_status, rd};
    c.tile_ctr = static_cast<unsigned int*>(ws);
    moe_status st = from_cuda(moe::launch_grouped_gemm(c, stream));
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

moe_status moe_grouped_gemm_fc2(const moe_bf16* h, const moe_bf16* wo,
                                const int32_t* group_offsets, moe_bf16* ys, int32_t* dev_status,
                                void* ws, moe_dims d, cudaStream_t stream) {
  (void)ws;
  MOE_CHECK_DIMS(d);
  MOE_OPTIONAL(dev_status);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(h);
  MOE_REQUIRE(wo);
  MOE_REQUIRE(group_offsets);
  MOE_REQUIRE(ys);
  GemmCall c{GemmKind::kFc2, h, wo, group_offsets, ys, nullptr, nullptr, dev_status, d};
  return from_cuda(moe::launch_grouped_gemm(c, stream));
}

moe_status moe_grouped_gemm_fc2_bwd(const moe_bf16* dys, const moe_bf16* h, const moe_bf16* wo,
                                    const moe_bf16* z, const int32_t* group_offsets,
                                    moe_bf16* dh_or_dz, moe_bf16* dwo, int32_t* dev_status,
                                    void* ws, moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(z);
  MOE_OPTIONAL(dh_or_dz);
  MOE_OPTIONAL(dwo);
  if (dh_or_dz == nullptr && dwo == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE(group_offsets);
  if (d.T > 0) {
    MOE_REQUIRE(dys);
    if (dh_or_dz != nullptr) MOE_REQUIRE(wo);
    if (dwo != nullptr) {
      MOE_REQUIRE(h);
      MOE_REQUIRE(ws);
    }
  }
  if (dh_or_dz != nullptr && d.T > 0) {
    GemmCall c{GemmKind::kDlhsFc2, dys, wo, group_offsets, dh_or_dz, nullptr, z, dev_status, d};
    moe_status st = from_cuda(moe::launch_grouped_gemm(c, stream));
    if (st != MOE_OK) return st;
  }
  if (dwo != nullptr) {
    GemmCall c{GemmKind::kDrhsFc2, h, dys, group_offsets, dwo, nullptr, nullptr, dev_status, d};
    c.tile_ctr = static_cast<unsigned int*>(ws);
    moe_status st = from_cuda(moe::launch_grouped_gemm(c, stream));
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

moe_status moe_grouped_gemm_fc1_swiglu_bwd(const moe_bf16* grad, const moe_bf16* z,
                                           const moe_bf16* xs, const moe_bf16* wi,
                                           const int32_t* group_offsets, moe_bf16* dxs,
                                           moe_bf16* dwi, int32_t* dev_status, void* ws,
                                           moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(z);
  MOE_OPTIONAL(dxs);
  MOE_OPTIONAL(dwi);
  if (dxs == nullptr && dwi == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE(group_offsets);
  const moe_bf16* dz = grad;
  if (d.T > 0) {
    MOE_REQUIRE(grad);
    if (dxs != nullptr) MOE_REQUIRE(wi);
    if (dwi != nullptr) {
      MOE_REQUIRE(xs);
      MOE_REQUIRE(ws);
    }
    if (z != nullptr) {
      // grad is dh [R,F]: the SwiGLU backward writes dz into the workspace,
      // after the bytes of the drhs tile counter
      MOE_REQUIRE(ws);
      moe_bf16* dzw = reinterpret_cast<moe_bf16*>(static_cast<char*>(ws) + moe::kWsCounterBytes);
      cudaError_t e = moe::launch_swiglu_bwd(grad, z, dzw, rows(d), d.F, stream);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      dz = dzw;
    }
  }
  if (dxs != nullptr && d.T > 0) {
    GemmCall c{GemmKind::kDlhsFc1, dz, wi, group_offsets, dxs, nullptr, nullptr, dev_status, d};
    moe_status st = from_cuda(moe::launch_grouped_gemm(c, stream));
    if (st != MOE_OK) return st;
  }
  if (dwi != nullptr) {
    GemmCall c{GemmKind::kDrhsFc1, xs, dz, group_offsets, dwi, nullptr, nullptr, dev_status, d};
    c.tile_ctr = static_cast<unsigned int*>(ws);
    moe_status st = from_cuda(moe::launch_grouped_gemm(c, stream));
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

size_t moe_mx_bytes(moe_dims d, moe_mx_buffer which) {
  if (check_dims(d) != MOE_OK) return 0;
  const size_t R = static_cast<size_t>(rows(d)), D = d.D, F = d.F, E = d.E;
  const size_t tiles = static_cast<size_t>(moe::mx_tile_bound(d));
  const size_t kbd = static_cast<size_t>(moe::mx_kblocks(d.D));
  const size_t kbf = static_cast<size_t>(moe::mx_kblocks(d.F));
  switch (which) {
    case MOE_MX_XQ: return R * D;
    case MOE_MX_XSC: return tiles * kbd * 512;
    case MOE_MX_WIQ: return E * 2 * F * D;
    case MOE_MX_WISC: return E * kbd * static_cast<size_t>(moe::mx_weight_row_blocks(2 * F)) * 512;
    case MOE_MX_WOQ: return E * D * F;
    case MOE_MX_WOSC: return E * kbf * static_cast<size_t>(moe::mx_weight_row_blocks(d.D)) * 512;
    case MOE_MX_HQ: return R * F;
    case MOE_MX_HSC: return tiles * kbf * 512;
    case MOE_MX_DYQ: return R * D;
    case MOE_MX_DYSC: return tiles * kbd * 512;
    case MOE_MX_DZQ: return R * 2 * F;
    case MOE_MX_DZSC: return tiles * static_cast<size_t>(moe::mx_kblocks(2L * d.F)) * 512;
    case MOE_MX_WIQ_BWD: return E * D * 2 * F;
    case MOE_MX_WISC_BWD:
      return E * static_cast<size_t>(moe::mx_kblocks(2L * d.F)) *
             static_cast<size_t>(moe::mx_weight_row_blocks(d.D)) * 512;
    case MOE_MX_WOQ_BWD: return E * F * D;
    case MOE_MX_WOSC_BWD:
      return E * kbd * static_cast<size_t>(moe::mx_weight_row_blocks(d.F)) * 512;
    case MOE_MX_XT:
    case MOE_MX_DYT: return D * static_cast<size_t>(moe::mx_token_cols(d));
    case MOE_MX_HT: return F * static_cast<size_t>(moe::mx_token_cols(d));
    case MOE_MX_DZT: return 2 * F * static_cast<size_t>(moe::mx_token_cols(d));
    case MOE_MX_XTSC:
    case MOE_MX_DYTSC: return tiles * static_cast<size_t>(moe::mx_weight_row_blocks(d.D)) * 512;
    case MOE_MX_HTSC: return tiles * static_cast<size_t>(moe::mx_weight_row_blocks(d.F)) * 512;
    case MOE_MX_DZTSC:
      return tiles * static_cast<size_t>(moe::mx_weight_row_blocks(2L * d.F)) * 512;
  }
  return 0;
}

namespace {
moe_status mx_quantize_weight(const moe_bf16* w, uint8_t* wq, uint8_t* wsc, uint8_t* wq_bwd,
                              uint8_t* wsc_bwd, int E, int Kd, int N, bool fc1,
                              cudaStream_t stream) {
  MOE_REQUIRE(w);
  MOE_OPTIONAL(wq);
  MOE_OPTIONAL(wsc);
  MOE_OPTIONAL(wq_bwd);
  MOE_OPTIONAL(wsc_bwd);
  if ((wq == nullptr) != (wsc == nullptr) || (wq_bwd == nullptr) != (wsc_bwd == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (wq == nullptr && wq_bwd == nullptr) return MOE_ERR_INVALID_ARG;
  return from_cuda(moe::launch_mx_quantize_weights(w, wq, wsc, wq_bwd, wsc_bwd, E, Kd, N, fc1,
                                                   stream));
}
}  // namespace

moe_status moe_mx_quantize_wi(const moe_bf16* wi, uint8_t* wq, uint8_t* wsc, uint8_t* wq_bwd,
                              uint8_t* wsc_bwd, moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  return mx_quantize_weight(wi, wq, wsc, wq_bwd, wsc_bwd, d.E, d.D, 2 * d.F, true, stream);
}

moe_status moe_mx_quantize_wo(const moe_bf16* wo, uint8_t* wq, uint8_t* wsc, uint8_t* wq_bwd,
                              uint8_t* wsc_bwd, moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  return mx_quantize_weight(wo, wq, wsc, wq_bwd, wsc_bwd, d.E, d.F, d.D, false, stream);
}

moe_status moe_mx_permute_quantize(const moe_bf16* x, const int32_t* pos,
                                   const int32_t* group_offsets, uint8_t* xq, uint8_t* xsc,
                                   moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(x);
  MOE_REQUIRE(pos);
  MOE_REQUIRE(group_offsets);
  MOE_REQUIRE(xq);
  MOE_REQUIRE(xsc);
  return from_cuda(moe::launch_mx_permute_quantize(x, pos, group_offsets, xq, xsc, d, stream));
}

moe_status moe_mx_grouped_gemm_fc1_swiglu(const uint8_t* xq, const uint8_t* xsc,
                                          const uint8_t* wq, const uint8_t* wsc,
                                          const int32_t* group_offsets, uint8_t* hq,
                                          uint8_t* hsc, moe_bf16* h, moe_bf16* z,
                                          int32_t* dev_status, moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(hq);
  MOE_OPTIONAL(hsc);
  MOE_OPTIONAL(h);
  MOE_OPTIONAL(z);
  if ((hq == nullptr) != (hsc == nullptr)) return MOE_ERR_INVALID_ARG;
  if (hq == nullptr && h == nullptr) return MOE_ERR_INVALID_ARG;
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(xq);
  MOE_REQUIRE(xsc);
  MOE_REQUIRE(wq);
  MOE_REQUIRE(wsc);
  MOE_REQUIRE(group_offsets);
  moe::MxGemmCall c{moe::MxKind::kFc1, xq, xsc, wq, wsc, group_offsets, hq, hsc, h, nullptr, z,
                    dev_status, d, 0, 0, 0};
  return from_cuda(moe::launch_mx_grouped_gemm(c, stream));
}

moe_status moe_mx_grouped_gemm_fc2(const uint8_t* hq, const uint8_t* hsc, const uint8_t* wq,
                                   const uint8_t* wsc, const int32_t* group_offsets,
                                   moe_bf16* ys, int32_t* dev_status, moe_dims d,
                                   cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  MOE_OPTIONAL(dev_status);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(hq);
  MOE_REQUIRE(hsc);
  MOE_REQUIRE(wq);
  MOE_REQUIRE(wsc);
  MOE_REQUIRE(group_offsets);
  MOE_REQUIRE(ys);
  moe::MxGemmCall c{moe::MxKind::kRows, hq, hsc, wq, wsc, group_offsets, nullptr, nullptr, ys,
                    nullptr, nullptr, dev_status, d, d.F, d.D, 0};
  return from_cuda(moe::launch_mx_grouped_gemm(c, stream));
}

moe_status moe_mx_combine_bwd(const moe_bf16* dout, const moe_bf16* ys, const float* w,
                              const int32_t* pos, const int32_t* group_offsets, moe_bf16* dys,
                              uint8_t* dyq, uint8_t* dysc, float* dw, moe_dims d,
                              cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(dout);
  MOE_REQUIRE(ys);
  MOE_REQUIRE(w);
  MOE_REQUIRE(pos);
  MOE_REQUIRE(group_offsets);
  MOE_REQUIRE(dys);
  MOE_REQUIRE(dyq);
  MOE_REQUIRE(dysc);
  MOE_REQUIRE(dw);
  return from_cuda(
      moe::launch_mx_combine_bwd(dout, ys, w, pos, group_offsets, dys, dyq, dysc, dw, d, stream));
}

moe_status moe_mx_quantize_rows(const moe_bf16* src, int C, const int32_t* group_offsets,
                                uint8_t* q, uint8_t* sc, moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (C != d.D && C != 2 * d.F) return MOE_ERR_INVALID_ARG;
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(src);
  MOE_REQUIRE(group_offsets);
  MOE_REQUIRE(q);
  MOE_REQUIRE(sc);
  return from_cuda(moe::launch_mx_quantize_rows(src, group_offsets, q, sc, C, d, stream));
}

moe_status moe_mx_quantize_tokens(const moe_bf16* src, const int32_t* row_src, int C,
                                  const int32_t* group_offsets, uint8_t* qt, uint8_t* sct,
                                  moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  if (C != d.D && C != d.F && C != 2 * d.F) return MOE_ERR_INVALID_ARG;
  MOE_OPTIONAL(row_src);
  if (d.T == 0) return MOE_OK;
  MOE_REQUIRE(src);
  MOE_REQUIRE(group_offsets);
  MOE_REQUIRE(qt);
  MOE_REQUIRE(sct);
  return from_cuda(
      moe::launch_mx_quantize_tokens(src, row_src, group_offsets, qt, sct, C, d, stream));
}

namespace {
// out bf16 [E, m, n] of an MX wgrad (zeros where no token reaches an expert)
moe_status mx_wgrad(const uint8_t* at, const uint8_t* atsc, const uint8_t* bt,
                    const uint8_t* btsc, const int32_t* group_offsets, moe_bf16* out, int m,
                    int n, int32_t* dev_status, const moe_dims& d, cudaStream_t stream) {
  if (d.T == 0)
    return from_cuda(cudaMemsetAsync(out, 0, static_cast<size_t>(d.E) * m * n * 2, stream));
  MOE_REQUIRE(at);
  MOE_REQUIRE(atsc);
  MOE_REQUIRE(bt);
  MOE_REQUIRE(btsc);
  moe::MxGemmCall c{moe::MxKind::kWgrad, at, atsc, bt, btsc, group_offsets, nullptr, nullptr, out,
                    nullptr, nullptr, dev_status, d, 0, n, m};
  return from_cuda(moe::launch_mx_grouped_gemm(c, stream));
}
}  // namespace

moe_status moe_mx_grouped_gemm_fc2_bwd(const uint8_t* dyq, const uint8_t* dysc,
                                       const uint8_t* woq, const uint8_t* wosc, const moe_bf16* z,
                                       const uint8_t* ht, const uint8_t* htsc,
                                       const uint8_t* dyt, const uint8_t* dytsc,
                                       const int32_t* group_offsets, moe_bf16* dz, moe_bf16* dwo,
                                       int32_t* dev_status, moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(dz);
  MOE_OPTIONAL(dwo);
  if (dz == nullptr && dwo == nullptr) return MOE_ERR_INVALID_ARG;
  if (dwo != nullptr && d.T > 0) MOE_REQUIRE(group_offsets);
  if (dz != nullptr && d.T > 0) {
    MOE_REQUIRE(dyq);
    MOE_REQUIRE(dysc);
    MOE_REQUIRE(woq);
    MOE_REQUIRE(wosc);
    MOE_REQUIRE(z);
    MOE_REQUIRE(group_offsets);
    moe::MxGemmCall c{moe::MxKind::kRowsSwigluBwd, dyq, dysc, woq, wosc, group_offsets, nullptr,
                      nullptr, dz, z, nullptr, dev_status, d, 0, 0, 0};
    moe_status st = from_cuda(moe::launch_mx_grouped_gemm(c, stream));
    if (st != MOE_OK) return st;
  }
  if (dwo != nullptr)
    return mx_wgrad(ht, htsc, dyt, dytsc, group_offsets, dwo, d.F, d.D, dev_status, d, stream);
  return MOE_OK;
}

moe_status moe_mx_grouped_gemm_fc1_bwd(const uint8_t* dzq, const uint8_t* dzsc,
                                       const uint8_t* wiq, const uint8_t* wisc,
                                       const uint8_t* xt, const uint8_t* xtsc,
                                       const uint8_t* dzt, const uint8_t* dztsc,
                                       const int32_t* group_offsets, moe_bf16* dxs, moe_bf16* dwi,
                                       int32_t* dev_status, moe_dims d, cudaStream_t stream) {
  MOE_CHECK_DIMS(d);
  MOE_OPTIONAL(dev_status);
  MOE_OPTIONAL(dxs);
  MOE_OPTIONAL(dwi);
  if (dxs == nullptr && dwi == nullptr) return MOE_ERR_INVALID_ARG;
  if (dwi != nullptr && d.T > 0) MOE_REQUIRE(group_offsets);
  if (dxs != nullptr && d.T > 0) {
    MOE_REQUIRE(dzq);
    MOE_REQUIRE(dzsc);
    MOE_REQUIRE(wiq);
    MOE_REQUIRE(wisc);
    MOE_REQUIRE(group_offsets);
    moe::MxGemmCall c{moe::MxKind::kRows, dzq, dzsc, wiq, wisc, group_offsets, nullptr, nullptr,
                      dxs, nullptr, nullptr, dev_status, d, 2 * d.F, d.D, 0};
    moe_status st = from_cuda(moe::launch_mx_grouped_gemm(c, stream));
    if (st != MOE_OK) return st;
  }
  if (dwi != nullptr)
    return mx_wgrad(xt, xtsc, dzt, dztsc, group_offsets, dwi, d.D, 2 * d.F, dev_status, d, stream);
  return MOE_OK;
}

moe_status moe_selftest_bounded_wait(int32_t* dev_status, uint64_t limit_ns, cudaStream_t stream) {
  MOE_REQUIRE(dev_status);
  if (limit_ns == 0 || limit_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;
  return from_cuda(moe::launch_bounded_wait_selftest(dev_status, limit_ns, stream));
}

}  // extern "C"
