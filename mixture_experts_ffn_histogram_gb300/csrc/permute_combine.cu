// Permute, combine and their backward passes: HBM-bound gathers and
// scatters of bf16 rows, one warp per token, 16-byte vector accesses.
//
// MaxText "MoE: fused TensorCore Pallas permute/combine kernels and
// split-expert wi layout for TPU v6e", Context item 1 and Commits table rows
// 1-2:
//   permute      xs[pos[t,k]] = x[t]: each token row is read once and stored
//                to its K expert-sorted rows; the unsorted [T*K, D] copy never
//                exists.
//   combine      out[t] = sum_k w[t,k] * ys[pos[t,k]] (unpermute + weighted
//                sum in one pass).
//   combine_bwd  dys[pos[t,k]] = w[t,k] * dout[t] (a permutation) and
//                dw[t,k] = <dout[t], ys[pos[t,k]]> (a per-slot reduction).
//   permute_bwd  the combine with unit weights.
// In the combine, the permute backward and the dys scatter each product and
// each sum is rounded separately (no fused multiply-add) in ascending slot
// order, so those results are reproducible bit for bit; dw is an fp32 dot
// product accumulated per lane and reduced across the warp.
#include "common.cuh"
#include "kernels.h"
#include "mx_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;  // 8 warps = 8 tokens per block pass
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

int grid_for_tokens(int T) {
  const int want = (T + kWarps - 1) / kWarps;
  const int cap = sm_count() * 16;  // ~8 resident blocks per SM, two waves
  return want < cap ? want : cap;
}

// Warps per token row for the gathers.  With few tokens one warp per row
// leaves the SMs with too few loads in flight, so a row is split into
// column slices of whole 32*VPL-vector passes, one warp each, until about
// `want_warps` warps are busy.  Every output element is still computed by
// one lane in the same order, so results do not change.
int split_for_tokens(int T, int Dv, int vpl, long want_warps) {
  const int max_split = max(1, Dv / (32 * vpl));
  long sp = T > 0 ? (want_warps + T - 1) / T : 1;
  if (sp < 1) sp = 1;
  if (sp > max_split) sp = max_split;
  return static_cast<int>(sp);
}
int grid_for_rows(int T, int split) {
  const long want = (static_cast<long>(T) * split + kWarps - 1) / kWarps;
  const long cap = static_cast<long>(sm_count()) * 16;
  return static_cast<int>(want < cap ? want : cap);
}

// VPL: 16-byte vectors per lane per pass; SPLIT: rows shared by `split`
// warps (a separate instantiation, so that one warp per row keeps its
// register count)
template <int VPL, bool SPLIT>
__global__ void __launch_bounds__(kThreads) permute_kernel(const uint4* __restrict__ x,
                                                           const int32_t* __restrict__ pos,
                                                           uint4* __restrict__ xs, int T, int K,
                                                           int Dv, int split_arg) {
  const int lane = threadIdx.x & 31;
  const int split = SPLIT ? split_arg : 1;
  const int passes = (Dv + 32 * VPL - 1) / (32 * VPL);  // 32*VPL-vector passes per row
  const int slice = (passes + split - 1) / split * (32 * VPL);  // vectors per slice
  const long items = static_cast<long>(T) * split;
  for (long u = static_cast<long>(blockIdx.x) * kWarps + (threadIdx.x >> 5); u < items;
       u += static_cast<long>(gridDim.x) * kWarps) {
    const int t = static_cast<int>(u / split);
    const int c0 = static_cast<int>(u - static_cast<long>(t) * split) * slice;
    const int c1 = min(Dv, c0 + slice);
    const int p_lane = (lane < K) ? __ldg(pos + static_cast<long>(t) * K + lane) : -1;
    const uint4* src = x + static_cast<long>(t) * Dv;
    for (int v0 = c0; v0 < c1; v0 += 32 * VPL) {
      uint4 buf[VPL];
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int idx = v0 + i * 32 + lane;
        if (idx < c1) buf[i] = ld_stream(src + idx);
      }
      for (int k = 0; k < K; ++k) {
        const int p = __shfl_sync(0xffffffffu, p_lane, k);
        if (p < 0) continue;
        uint4* dst = xs + static_cast<long>(p) * Dv;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int idx = v0 + i * 32 + lane;
          if (idx < c1) dst[idx] = buf[i];
        }
      }
    }
  }
}

__device__ __forceinline__ void axpy8(float (&acc)[8], float wk, const uint4& v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] = __fadd_rn(acc[2 * q], __fmul_rn(wk, bf16lo(u[q])));
    acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __fmul_rn(wk, bf16hi(u[q])));
  }
}

// Slots of the combine backward whose ys rows one lane has in flight at once:
// their loads are issued before any of them is used, so a warp waits for one
// DRAM round trip per batch instead of one per slot (measured at the
// long-sequence shape: 522 -> 474 us).  The forward gather is the opposite
// case: there one slot at a time beat batches of 2, 4 and 8 slots at every
// measured shape (long sequence, 8192 and 1024 tokens), and more warps per
// row are what helps when tokens are few.
constexpr int kSlotBatch = 8;

// out[t] = bf16(sum_k w[t,k] * ys[pos[t,k]]); w == nullptr means unit weights.
template <int VPL, bool SPLIT>
__global__ void __launch_bounds__(kThreads) combine_kernel(const uint4* __restrict__ ys,
                                                           const float* __restrict__ w,
                                                           const int32_t* __restrict__ pos,
                                                           uint4* __restrict__ out, int T, int K,
                                                           int Dv, int split_arg) {
  const int lane = threadIdx.x & 31;
  const int split = SPLIT ? split_arg : 1;
  const int passes = (Dv + 32 * VPL - 1) / (32 * VPL);  // 32*VPL-vector passes per row
  const int slice = (passes + split - 1) / split * (32 * VPL);  // vectors per slice
  const long items = static_cast<long>(T) * split;
  for (long u = static_cast<long>(blockIdx.x) * kWarps + (threadIdx.x >> 5); u < items;
       u += static_cast<long>(gridDim.x) * kWarps) {
    const int t = static_cast<int>(u / split);
    const int c0 = static_cast<int>(u - static_cast<long>(t) * split) * slice;
    const int c1 = min(Dv, c0 + slice);
    const long j = static_cast<long>(t) * K + lane;
    const int p_lane = (lane < K) ? __ldg(pos + j) : -1;
    const float w_lane = (lane < K) ? (w != nullptr ? __ldg(w + j) : 1.0f) : 0.f;
    for (int v0 = c0; v0 < c1; v0 += 32 * VPL) {
      float acc[VPL][8];
#pragma unroll
      for (int i = 0; i < VPL; ++i)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[i][q] = 0.f;
      for (int k = 0; k < K; ++k) {
        const int p = __shfl_sync(0xffffffffu, p_lane, k);
        const float wk = __shfl_sync(0xffffffffu, w_lane, k);
        if (p < 0) continue;
        const uint4* src = ys + static_cast<long>(p) * Dv;
        uint4 v[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int idx = v0 + i * 32 + lane;
          if (idx < c1) v[i] = ld_stream(src + idx);
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i) axpy8(acc[i], wk, v[i]);
      }
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int idx = v0 + i * 32 + lane;
        if (idx < c1) {
          uint4 o;
          o.x = pack_bf16x2(acc[i][0], acc[i][1]);
          o.y = pack_bf16x2(acc[i][2], acc[i][3]);
          o.z = pack_bf16x2(acc[i][4], acc[i][5]);
          o.w = pack_bf16x2(acc[i][6], acc[i][7]);
          out[static_cast<long>(t) * Dv + idx] = o;
        }
      }
    }
  }
}

// dys[pos[t,k]] = bf16(w * dout[t]);  dw[t,k] = <dout[t], ys[pos[t,k]]>.
// Slots go in batches of kSlotBatch: per column chunk, the dout vectors and
// the ys vectors of every slot of the batch are loaded before any is used.
// Each lane accumulates its part of a dot product over the chunks in
// ascending column order; the warp then sums the lanes' parts.
// With QUANT, each dys row is also quantized along D as MXFP8 for the FC2
// dgrad (moe_mx_combine_bwd): four consecutive lanes hold one 32-element
// block (their 16-byte vectors), whose largest magnitude two shuffles
// gather; each lane writes its 8 codes (a warp, 256 contiguous bytes) and
// the block's first lane its scale byte, in the tile-blocked layout of the
// row's group (the offsets and tile bases staged in shared memory).
struct MxRowsOut {
  const int32_t* offs;  // group offsets [E+1]
  uint8_t* q;           // codes [R][D]
  uint8_t* sc;          // tile-blocked scales
  int E;
  int KB;               // k-blocks of D
};

template <int VPL, bool QUANT>
__global__ void __launch_bounds__(kThreads, 2) combine_bwd_kernel(
    const uint4* __restrict__ dout, const uint4* __restrict__ ys, const float* __restrict__ w,
    const int32_t* __restrict__ pos, uint4* __restrict__ dys, float* __restrict__ dw, int T, int K,
    int Dv, MxRowsOut mq) {
  const int lane = threadIdx.x & 31;
  extern __shared__ int cb_bases[];  // QUANT: group offsets and tile bases
  if constexpr (QUANT) load_tile_bases(mq.offs, mq.E, cb_bases, cb_bases + mq.E + 1, 0);
  for (int t = blockIdx.x * kWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kWarps) {
    const long j = static_cast<long>(t) * K + lane;
    const int p_lane = (lane < K) ? __ldg(pos + j) : -1;
    const float w_lane = (lane < K) ? __ldg(w + j) : 0.f;
    const uint4* g = dout + static_cast<long>(t) * Dv;
    // (the quantizing variant takes half the batch: two blocks per SM need
    // its registers)
    constexpr int kBatch = QUANT ? kSlotBatch / 2 : kSlotBatch;
    for (int k0 = 0; k0 < K; k0 += kBatch) {
      int pk[kBatch];
      float wk[kBatch], dot[kBatch];
      size_t sbase[kBatch];  // QUANT: the row's first scale block (bytes)
      int sm[kBatch];        // QUANT: the row's place in its 128-row tile
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int k = k0 + b;
        pk[b] = (k < K) ? __shfl_sync(0xffffffffu, p_lane, k) : -1;
        wk[b] = (k < K) ? __shfl_sync(0xffffffffu, w_lane, k) : 0.f;
        dot[b] = 0.f;
        if constexpr (QUANT) {
          sbase[b] = 0;
          sm[b] = 0;
          if (pk[b] >= 0) {
            const int* s_off = cb_bases;
            const int* s_tb = cb_bases + mq.E + 1;
            const int e = group_of_row(s_off, mq.E, pk[b]);
            const int i = pk[b] - s_off[e];
            sbase[b] = static_cast<size_t>(s_tb[e] + (i >> 7)) * mq.KB * 512;
            sm[b] = i & 127;
          }
        }
      }
      for (int v0 = 0; v0 < Dv; v0 += 32 * VPL) {
        uint4 gv[VPL], yv[kBatch][VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int idx = v0 + i * 32 + lane;
          if (idx < Dv) gv[i] = __ldg(g + idx);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          if (pk[b] < 0) continue;
          const uint4* y = ys + static_cast<long>(pk[b]) * Dv;
#pragma unroll
          for (int i = 0; i < VPL; ++i) {
            const int idx = v0 + i * 32 + lane;
            if (idx < Dv) yv[b][i] = ld_stream(y + idx);
          }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          if (pk[b] < 0) continue;
          uint4* dst = dys + static_cast<long>(pk[b]) * Dv;
#pragma unroll
          for (int i = 0; i < VPL; ++i) {
            const int idx = v0 + i * 32 + lane;
            if (idx < Dv) {
              const uint32_t gu[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
              const uint32_t yu[4] = {yv[b][i].x, yv[b][i].y, yv[b][i].z, yv[b][i].w};
              uint32_t o[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float g0 = bf16lo(gu[q]), g1 = bf16hi(gu[q]);
                o[q] = pack_bf16x2(__fmul_rn(wk[b], g0), __fmul_rn(wk[b], g1));
                dot[b] = fmaf(g0, bf16lo(yu[q]), dot[b]);
                dot[b] = fmaf(g1, bf16hi(yu[q]), dot[b]);
              }
              dst[idx] = make_uint4(o[0], o[1], o[2], o[3]);
              if constexpr (QUANT) {
                // the bf16 values just stored, quantized in blocks of 4 lanes
                // (Dv % 4 == 0: a block's lanes are all in range together)
                float amax = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  amax = fmaxf(amax, fmaxf(fabsf(bf16lo(o[q])), fabsf(bf16hi(o[q]))));
                amax = fmaxf(amax, __shfl_xor_sync(0x0000000Fu << (lane & 28), amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0x0000000Fu << (lane & 28), amax, 2));
                const int sx = mx_shared_exp(amax);
                const float mul = mx_inv_scale(sx);
                const uint32_t c0 = e4m3x2(bf16lo(o[0]) * mul, bf16hi(o[0]) * mul);
                const uint32_t c1 = e4m3x2(bf16lo(o[1]) * mul, bf16hi(o[1]) * mul);
                const uint32_t c2 = e4m3x2(bf16lo(o[2]) * mul, bf16hi(o[2]) * mul);
                const uint32_t c3 = e4m3x2(bf16lo(o[3]) * mul, bf16hi(o[3]) * mul);
                *reinterpret_cast<uint2*>(mq.q + static_cast<size_t>(pk[b]) * Dv * 8 + idx * 8) =
                    make_uint2(__byte_perm(c0, c1, 0x5410), __byte_perm(c2, c3, 0x5410));
                if ((lane & 3) == 0) {
                  const int blk = idx >> 2;  // 32-element block along D
                  mq.sc[sbase[b] + static_cast<size_t>(blk >> 2) * 512 + sf_byte(sm[b], blk & 3)] =
                      static_cast<uint8_t>(sx + 127);
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        float d = dot[b];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        if (lane == 0 && k0 + b < K) dw[static_cast<long>(t) * K + k0 + b] = d;
      }
    }
  }
}

// dz = [dgate | dup] from a stored bf16 dh [R,F] and z [R,2F] (the SwiGLU
// backward of MaxText "Gemma4 26B MoE on TPU v6e", Commits table row 7,
// written as one tensor).  One thread per 8 columns.
__global__ void __launch_bounds__(kThreads) swiglu_bwd_kernel(const uint4* __restrict__ dh,
                                                              const uint4* __restrict__ z,
                                                              uint4* __restrict__ dz, long R,
                                                              int Fv) {
  const long n = R * Fv;
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const long r = i / Fv;
    const int c = static_cast<int>(i - r * Fv);
    const uint4 hv = __ldg(dh + i);
    const uint4 gv = __ldg(z + r * 2 * Fv + c);
    const uint4 uv = __ldg(z + r * 2 * Fv + Fv + c);
    const uint32_t hu[4] = {hv.x, hv.y, hv.z, hv.w};
    const uint32_t gu[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t uu[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t og[4], ou[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float dg[2], du[2];
#pragma unroll
      for (int hcomp = 0; hcomp < 2; ++hcomp) {
        const float d = hcomp ? bf16hi(hu[q]) : bf16lo(hu[q]);
        const float g = hcomp ? bf16hi(gu[q]) : bf16lo(gu[q]);
        const float u = hcomp ? bf16hi(uu[q]) : bf16lo(uu[q]);
        const float s = 1.0f / (1.0f + expf(-g));
        dg[hcomp] = d * u * s * (1.0f + g * (1.0f - s));
        du[hcomp] = d * g * s;
      }
      og[q] = pack_bf16x2(dg[0], dg[1]);
      ou[q] = pack_bf16x2(du[0], du[1]);
    }
    dz[r * 2 * Fv + c] = make_uint4(og[0], og[1], og[2], og[3]);
    dz[r * 2 * Fv + Fv + c] = make_uint4(ou[0], ou[1], ou[2], ou[3]);
  }
}

// out = bf16(acc), 8 elements per thread (the fused forward's last step).
__global__ void __launch_bounds__(kThreads) acc_to_bf16_kernel(const float4* __restrict__ acc,
                                                               uint4* __restrict__ out, long n8) {
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(acc + 2 * i), b = __ldg(acc + 2 * i + 1);
    out[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                        pack_bf16x2(b.z, b.w));
  }
}

// A block that waits on a barrier nothing arrives at, to exercise the
// bounded wait: it must give up, record MOE_ERR_TIMEOUT and return.
__global__ void bounded_wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  WaitCtl c{&abort_flag, status, limit_ns};
  if (threadIdx.x < 32) (void)mbar_wait(&bar, 0, c);
  __syncthreads();
}

}  // namespace

cudaError_t launch_permute(const uint16_t* x, const int32_t* pos, uint16_t* xs, const moe_dims& d,
                           cudaStream_t s) {
  if (d.T == 0) return cudaSuccess;
  const int split = split_for_tokens(d.T, d.D / 8, 4, static_cast<long>(sm_count()) * 64);
  auto kern = split > 1 ? permute_kernel<4, true> : permute_kernel<4, false>;
  kern<<<grid_for_rows(d.T, split), kThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(x), pos, reinterpret_cast<uint4*>(xs), d.T, d.K, d.D / 8,
      split);
  return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* ys, const float* w, const int32_t* pos, uint16_t* out,
                           const moe_dims& d, cudaStream_t s) {
  if (d.T == 0) return cudaSuccess;
  // measured on GB300: from 16384 tokens one warp per row with 4 vectors per
  // lane (long sequence, 32768 tokens: 271 vs 284 us with 2); below, rows
  // split until ~16384 warps run (8192 tokens: 57 vs 65 us unsplit; 1024
  // tokens: 14 vs 28 us)
  const auto* src = reinterpret_cast<const uint4*>(ys);
  auto* dst = reinterpret_cast<uint4*>(out);
  const int Dv = d.D / 8;
  if (d.T >= 16384) {
    combine_kernel<4, false><<<grid_for_rows(d.T, 1), kThreads, 0, s>>>(src, w, pos, dst, d.T,
                                                                             d.K, Dv, 1);
    return cudaGetLastError();
  }
  const int split = split_for_tokens(d.T, Dv, 2, 16384);
  auto kern = split > 1 ? combine_kernel<2, true> : combine_kernel<2, false>;
  kern<<<grid_for_rows(d.T, split), kThreads, 0, s>>>(src, w, pos, dst, d.T, d.K, Dv, split);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const uint16_t* dout, const uint16_t* ys, const float* w,
                               const int32_t* pos, uint16_t* dys, float* dw, const moe_dims& d,
                               cudaStream_t s) {
  if (d.T == 0) return cudaSuccess;
  combine_bwd_kernel<2, false><<<grid_for_tokens(d.T), kThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(dout), reinterpret_cast<const uint4*>(ys), w, pos,
      reinterpret_cast<uint4*>(dys), dw, d.T, d.K, d.D / 8, MxRowsOut{});
  return cudaGetLastError();
}

cudaError_t launch_mx_combine_bwd(const uint16_t* dout, const uint16_t* ys, const float* w,
                                  const int32_t* pos, const int32_t* offs, uint16_t* dys,
                                  uint8_t* dyq, uint8_t* dysc, float* dw, const moe_dims& d,
                                  cudaStream_t s) {
  if (d.T == 0) return cudaSuccess;
  const MxRowsOut mq{offs, dyq, dysc, d.E, (d.D + 127) / 128};
  combine_bwd_kernel<2, true><<<grid_for_tokens(d.T), kThreads, 8 * (d.E + 1), s>>>(
      reinterpret_cast<const uint4*>(dout), reinterpret_cast<const uint4*>(ys), w, pos,
      reinterpret_cast<uint4*>(dys), dw, d.T, d.K, d.D / 8, mq);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const uint16_t* dh, const uint16_t* z, uint16_t* dz, long R, int F,
                              cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const long n = R * (F / 8);
  long blocks = (n + kThreads - 1) / kThreads;
  const long cap = static_cast<long>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  swiglu_bwd_kernel<<<static_cast<int>(blocks), kThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(dh), reinterpret_cast<const uint4*>(z),
      reinterpret_cast<uint4*>(dz), R, F / 8);
  return cudaGetLastError();
}

cudaError_t launch_acc_to_bf16(const float* acc, uint16_t* out, long n, cudaStream_t s) {
  const long n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  long blocks = (n8 + kThreads - 1) / kThreads;
  const long cap = static_cast<long>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  acc_to_bf16_kernel<<<static_cast<int>(blocks), kThreads, 0, s>>>(
      reinterpret_cast<const float4*>(acc), reinterpret_cast<uint4*>(out), n8);
  return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(int32_t* dev_status, uint64_t limit_ns, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 64, 0, s>>>(dev_status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
