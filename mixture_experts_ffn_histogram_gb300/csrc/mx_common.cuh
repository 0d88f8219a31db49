// Device helpers of the MXFP8 kernels (OCP MX v1.0 MXFP8, as read for
// TransformerEngine "[DRAFT][JAX] Optimize MoE block", Changes item 1:
// blocks of 32 elements share an E8M0 scale 2^s, s = max(floor(log2 amax)
// - 8, -127); elements are E4M3 codes of v / 2^s, nearest-even, saturating),
// shared by mx.cu and the fused MX combine backward in permute_combine.cu.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// ------------------------------------------------------------ MX helpers
// Shared exponent of a block from its largest magnitude: floor(log2 amax) - 8
// from the fp32 exponent field, -127 for zero and fp32 subnormals (whose
// floor(log2) - 8 lies below -127 anyway).
__device__ __forceinline__ int mx_shared_exp(float amax) {
  const int be = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  if (be == 0) return -127;
  return max(be - 127 - 8, -127);
}
// 2^-s as an fp32 (s in [-127, 119], so 127 - s is a normal exponent)
__device__ __forceinline__ float mx_inv_scale(int s) {
  return __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
}
// Codes of 32 values (already multiplied by 2^-s), packed little-endian.
__device__ __forceinline__ void mx_pack32(const float (&v)[32], float mul, uint32_t (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i] * mul, v[4 * i + 1] * mul),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(v[4 * i + 2] * mul, v[4 * i + 3] * mul), __NV_SATFINITE, __NV_E4M3);
    w[i] = (lo & 0xFFFFu) | (hi << 16);
  }
}
// Quantize 32 values: codes into w, returns the scale byte.
__device__ __forceinline__ uint32_t mx_quant32(const float (&v)[32], uint32_t (&w)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int s = mx_shared_exp(amax);
  mx_pack32(v, mx_inv_scale(s), w);
  return static_cast<uint32_t>(s + 127);
}
// Byte of row m (0..127) and 32-element step j (0..3) inside a 512-byte
// scale block.
__device__ __forceinline__ int sf_byte(int m, int j) { return (m & 31) * 16 + (m >> 5) * 4 + j; }

// Shared exponent from the 8-bit exponent field of a block's largest
// magnitude (bf16 and fp32 share it): floor(log2 amax) - 8, -127 for zero
// and subnormals.
__device__ __forceinline__ int mx_exp_field(uint32_t ef) {
  return ef == 0 ? -127 : max(static_cast<int>(ef) - 127 - 8, -127);
}
// Two codes (low byte first) of two fp32 values already scaled.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3) & 0xFFFFu;
}
// MX blocks of two columns at once: w[i] holds row i of column A (low bf16)
// and of column B (high bf16), i = 0..31.  The largest magnitudes come from
// a per-halfword unsigned max of the sign-cleared bf16 bits (magnitude order
// is the unsigned order of those bits).  Returns the two scale bytes (A in
// bits 0-7, B in 8-15); ca/cb get the 32 codes of each column in row order.
__device__ __forceinline__ uint32_t mx_quant_col2(const uint32_t (&w)[32], uint32_t (&ca)[8],
                                                  uint32_t (&cb)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
  const int sa = mx_exp_field((m >> 7) & 0xFFu), sb = mx_exp_field((m >> 23) & 0xFFu);
  const float ma = mx_inv_scale(sa), mb = mx_inv_scale(sb);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t* r = w + 4 * i;
    const uint32_t a01 = e4m3x2(__uint_as_float(r[0] << 16) * ma, __uint_as_float(r[1] << 16) * ma);
    const uint32_t a23 = e4m3x2(__uint_as_float(r[2] << 16) * ma, __uint_as_float(r[3] << 16) * ma);
    const uint32_t b01 = e4m3x2(__uint_as_float(r[0] & 0xFFFF0000u) * mb,
                                __uint_as_float(r[1] & 0xFFFF0000u) * mb);
    const uint32_t b23 = e4m3x2(__uint_as_float(r[2] & 0xFFFF0000u) * mb,
                                __uint_as_float(r[3] & 0xFFFF0000u) * mb);
    ca[i] = __byte_perm(a01, a23, 0x5410);
    cb[i] = __byte_perm(b01, b23, 0x5410);
  }
  return static_cast<uint32_t>(sa + 127) | (static_cast<uint32_t>(sb + 127) << 8);
}
// One MX block of 32 consecutive bf16 (w[i] = elements 2i, 2i+1): codes and
// the scale byte.
__device__ __forceinline__ uint32_t mx_quant_row32(const uint32_t (&w)[16], uint32_t (&c)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
  m = max(m & 0xFFFFu, m >> 16);
  const int s = mx_exp_field((m >> 7) & 0xFFu);
  const float mul = mx_inv_scale(s);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = e4m3x2(__uint_as_float(w[2 * i] << 16) * mul,
                               __uint_as_float(w[2 * i] & 0xFFFF0000u) * mul);
    const uint32_t hi = e4m3x2(__uint_as_float(w[2 * i + 1] << 16) * mul,
                               __uint_as_float(w[2 * i + 1] & 0xFFFF0000u) * mul);
    c[i] = __byte_perm(lo, hi, 0x5410);
  }
  return static_cast<uint32_t>(s + 127);
}

// Group offsets into shared memory (all threads), then the exclusive prefix
// of ceil(rows/128) over the groups (one warp).  Ends with __syncthreads().
__device__ __forceinline__ void load_tile_bases(const int32_t* offs, int E, int* s_off, int* s_tb,
                                                int scan_warp) {
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = __ldg(offs + i);
  __syncthreads();
  if (static_cast<int>(threadIdx.x >> 5) == scan_warp) {
    const int lane = threadIdx.x & 31;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int local = 0;
    for (int e = e0; e < e1; ++e) local += (s_off[e + 1] - s_off[e] + 127) >> 7;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e1; ++e) {
      s_tb[e] = run;
      run += (s_off[e + 1] - s_off[e] + 127) >> 7;
    }
    if (lane == 31) s_tb[E] = incl;
  }
  __syncthreads();
}

// Group of sorted row r: the largest e with s_off[e] <= r (r < s_off[E]).
__device__ __forceinline__ int group_of_row(const int* s_off, int E, int r) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_off[mid] <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

}  // namespace moe
