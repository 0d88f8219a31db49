/*
 * CPU oracle for the sparse MoE expert block -- TEST INFRASTRUCTURE ONLY.
 * (See oracle.h for who may use it and for the conventions.)
 *
 * This file writes out the plain definition of each step of the block, one
 * function per entry point of the CUDA library, in the order and notation of
 * the pages it follows:
 *
 *   [Keep fused]  MaxText "Keep fused MoE weights intact through FSDP gather",
 *                 Description (updated flow: one grouped GEMM on the prefused
 *                 [experts, embed, 2*mlp] weight, then split the output
 *                 activations for SwiGLU).
 *   [Fused p/c]   MaxText "MoE: fused TensorCore Pallas permute/combine
 *                 kernels and split-expert wi layout for TPU v6e", Context
 *                 item 1 and Commits table rows 1-2 (combine = unpermute +
 *                 top-K weighted sum; its backward = a permutation for dx and
 *                 a per-slot reduction for dw; permute = gather into expert-
 *                 sorted order with the group_size histogram computed first;
 *                 permute backward = combine with unit weights) and Tests
 *                 (f32 routing weights).
 *   [Gemma4 L/M]  MaxText "Gemma4 26B MoE on TPU v6e: MaxText layer/model
 *                 optimizations", Commits table row 6 (top_k_weights and
 *                 group_size), row 7 and the code-review suggestion
 *                 (_split_gate_up_bwd: the gate/up gradient is one
 *                 concatenation [grad_gate, grad_up] along the last axis).
 *   [TE MoE]      TransformerEngine "[DRAFT][JAX] Optimize MoE block",
 *                 Flowchart (routing -> grouped FC1 -> activation and
 *                 grouped FC2 -> combine).
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes):  top-K ties go to the lower expert id; the expert-sorted order is
 * stable in the flat slot index t*K+k; gate = columns [0,F) of wi's last
 * axis and up = [F,2F); bf16 rounding exactly where a tensor is stored; the
 * block is dropless.
 *
 * Parity pins: every function here is checked against brute force, library
 * routines, closed forms, finite differences and invariants by the CPU test
 * suite; none is "parity unpinned".
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
  /* round to nearest, ties to even, on the 16 discarded bits */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

#define BF(b) oracle_bf16_to_f32(b)
#define RN(f) oracle_f32_to_bf16(f)

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static float sigmoidf_(float v) { return 1.0f / (1.0f + expf(-v)); }

/* Step 1, routing [Gemma4 L/M row 6]: per token, the K largest scores in
 * descending order (ties: lower expert id first), and their weights:
 *   SOFTMAX_TOPK: w_k = exp(s_k - s_0) / sum_j exp(s_j - s_0) over the K selected;
 *   SIGMOID_NORM: w_k = sigmoid(s_k) / sum_j sigmoid(s_j) over the K selected;
 * with s = logit (+ bias[e] when a bias is given).  GIVEN: ids/w are inputs. */
int oracle_route(const float* logits, const float* bias, int mode, int T, int E, int K,
                 int32_t* ids, float* w) {
  if (T < 0 || E <= 0 || K <= 0 || K > E) return -1;
  if (mode == ORACLE_GIVEN) return 0;
  if (mode != ORACLE_SOFTMAX_TOPK && mode != ORACLE_SIGMOID_NORM) return -1;
  int bad = 0;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
    unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
    for (int e = 0; e < E; ++e) {
      float v = logits[(size_t)t * E + e];
      s[e] = bias ? v + bias[e] : v;
    }
    for (int k = 0; k < K; ++k) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || s[e] > s[best]) best = e;  /* strict: ties keep the lower id */
      }
      taken[best] = 1;
      ids[(size_t)t * K + k] = best;
    }
    float sum = 0.0f;
    float* v = w + (size_t)t * K;
    if (mode == ORACLE_SOFTMAX_TOPK) {
      float m = s[ids[(size_t)t * K]];
      for (int k = 0; k < K; ++k) { v[k] = expf(s[ids[(size_t)t * K + k]] - m); sum = sum + v[k]; }
    } else {
      for (int k = 0; k < K; ++k) { v[k] = sigmoidf_(s[ids[(size_t)t * K + k]]); sum = sum + v[k]; }
    }
    for (int k = 0; k < K; ++k) v[k] = v[k] / sum;
    free(s);
    free(taken);
  }
  return bad;
}

/* Step 2, group_size histogram above the gather [Fused p/c row 2; Gemma4 L/M
 * row 6]: flatten ids token-major (j = t*K + k);
 *   group_sizes[e] = #{j : ids[j] = e};  group_offsets = exclusive prefix sum;
 *   pos[j] = group_offsets[ids[j]] + #{j' < j : ids[j'] = ids[j]}  (stable);
 *   row_src[pos[j]] = j.
 * Slots whose id lies outside [0,E) get pos = -1 and are not counted; the
 * rows left over at the end of row_src are -1.  Returns that slot count. */
int oracle_histogram(const int32_t* ids, int T, int K, int E, int32_t* group_sizes,
                     int32_t* group_offsets, int32_t* pos, int32_t* row_src) {
  if (T < 0 || K <= 0 || E <= 0) return -1;
  const long R = (long)T * K;
  int bad = 0;
  for (int e = 0; e < E; ++e) group_sizes[e] = 0;
  for (long j = 0; j < R; ++j) {
    int e = ids[j];
    if (e < 0 || e >= E) { ++bad; continue; }
    group_sizes[e] += 1;
  }
  group_offsets[0] = 0;
  for (int e = 0; e < E; ++e) group_offsets[e + 1] = group_offsets[e] + group_sizes[e];
  int32_t* seen = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (long j = 0; j < R; ++j) row_src[j] = -1;
  for (long j = 0; j < R; ++j) {
    int e = ids[j];
    if (e < 0 || e >= E) { pos[j] = -1; continue; }
    int p = group_offsets[e] + seen[e];
    seen[e] += 1;
    pos[j] = p;
    row_src[p] = (int32_t)j;
  }
  free(seen);
  return bad;
}

/* Step 3, permute [Fused p/c Context 1, row 2]: xs[pos[t,k]] = x[t] (exact). */
int oracle_permute(const uint16_t* x, const int32_t* pos, int T, int K, int D, uint16_t* xs) {
  if (T < 0 || K <= 0 || D <= 0) return -1;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int p = pos[(size_t)t * K + k];
      if (p < 0) continue;
      memcpy(xs + (size_t)p * D, x + (size_t)t * D, sizeof(uint16_t) * (size_t)D);
    }
  return 0;
}

/* Step 4, FC1 + SwiGLU [Keep fused, Description; TE MoE, Flowchart]: for
 * every row r of group e, a[n] = sum_d xs[r,d] * wi[e,d,n] over the whole
 * prefused weight (n < 2F), then g = a[0:F], u = a[F:2F],
 *   h[r,f] = bf16(silu(g_f) * u_f),  silu(g) = g * sigmoid(g);
 *   z[r,n] = bf16(a[n])  (stored for the backward when z != NULL). */
int oracle_fc1_swiglu(const uint16_t* xs, const uint16_t* wi, const int32_t* offs, int E,
                      int D, int F, uint16_t* h, uint16_t* z) {
  if (E <= 0 || D <= 0 || F <= 0) return -1;
  const int N = 2 * F;
  const int R = offs[E];
#pragma omp parallel
  {
    float* a = (float*)malloc(sizeof(float) * (size_t)N);
#pragma omp for schedule(dynamic, 4)
    for (int r = 0; r < R; ++r) {
      int e = 0;
      while (offs[e + 1] <= r) ++e;
      const uint16_t* W = wi + (size_t)e * D * N;
      for (int n = 0; n < N; ++n) a[n] = 0.0f;
      for (int d = 0; d < D; ++d) {
        float xv = BF(xs[(size_t)r * D + d]);
        const uint16_t* wr = W + (size_t)d * N;
        for (int n = 0; n < N; ++n) a[n] = a[n] + xv * BF(wr[n]);
      }
      for (int f = 0; f < F; ++f) {
        float g = a[f], u = a[F + f];
        h[(size_t)r * F + f] = RN((g * sigmoidf_(g)) * u);
      }
      if (z)
        for (int n = 0; n < N; ++n) z[(size_t)r * N + n] = RN(a[n]);
    }
    free(a);
  }
  return 0;
}

/* Step 5, FC2 [TE MoE, Flowchart]: ys[r,:] = bf16(sum_f h[r,f] * wo[e,f,:]). */
int oracle_fc2(const uint16_t* h, const uint16_t* wo, const int32_t* offs, int E, int F, int D,
               uint16_t* ys) {
  if (E <= 0 || D <= 0 || F <= 0) return -1;
  const int R = offs[E];
#pragma omp parallel
  {
    float* a = (float*)malloc(sizeof(float) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
    for (int r = 0; r < R; ++r) {
      int e = 0;
      while (offs[e + 1] <= r) ++e;
      const uint16_t* W = wo + (size_t)e * F * D;
      for (int d = 0; d < D; ++d) a[d] = 0.0f;
      for (int f = 0; f < F; ++f) {
        float hv = BF(h[(size_t)r * F + f]);
        const uint16_t* wr = W + (size_t)f * D;
        for (int d = 0; d < D; ++d) a[d] = a[d] + hv * BF(wr[d]);
      }
      for (int d = 0; d < D; ++d) ys[(size_t)r * D + d] = RN(a[d]);
    }
    free(a);
  }
  return 0;
}

/* Step 6, combine [Fused p/c row 1]: unpermute plus the top-K weighted sum,
 *   out[t] = bf16(sum_{k ascending} w[t,k] * ys[pos[t,k]]). */
int oracle_combine(const uint16_t* ys, const float* w, const int32_t* pos, int T, int K, int D,
                   uint16_t* out) {
  if (T < 0 || K <= 0 || D <= 0) return -1;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int d = 0; d < D; ++d) {
      float acc = 0.0f;
      for (int k = 0; k < K; ++k) {
        int p = pos[(size_t)t * K + k];
        if (p < 0) continue;
        float wk = w ? w[(size_t)t * K + k] : 1.0f;
        acc = acc + wk * BF(ys[(size_t)p * D + d]);
      }
      out[(size_t)t * D + d] = RN(acc);
    }
  return 0;
}

/* Backward of the combine [Fused p/c row 1: a permutation for dx and a
 * per-slot reduction for dw]:
 *   dys[pos[t,k]] = bf16(w[t,k] * dout[t]);
 *   dw[t,k] = sum_d dout[t,d] * ys[pos[t,k], d]  (fp32). */
int oracle_combine_bwd(const uint16_t* dout, const uint16_t* ys, const float* w,
                       const int32_t* pos, int T, int K, int D, uint16_t* dys, float* dw) {
  if (T < 0 || K <= 0 || D <= 0) return -1;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int p = pos[(size_t)t * K + k];
      if (p < 0) { dw[(size_t)t * K + k] = 0.0f; continue; }
      float wk = w[(size_t)t * K + k];
      float acc = 0.0f;
      for (int d = 0; d < D; ++d) {
        float g = BF(dout[(size_t)t * D + d]);
        dys[(size_t)p * D + d] = RN(wk * g);
        acc = acc + g * BF(ys[(size_t)p * D + d]);
      }
      dw[(size_t)t * K + k] = acc;
    }
  return 0;
}

/* SwiGLU backward at one element [Gemma4 L/M row 7 and review suggestion]:
 * with s = sigmoid(g), h = g*s*u:
 *   dgate = dh * u * s * (1 + g*(1 - s)),  dup = dh * g * s,
 * and dz = [dgate | dup] written as one [R, 2F] tensor (a concatenation). */
static void swiglu_bwd_one(float dh, float g, float u, float* dgate, float* dup) {
  float s = sigmoidf_(g);
  *dgate = ((dh * u) * s) * (1.0f + g * (1.0f - s));
  *dup = (dh * g) * s;
}

/* Backward of FC2: dlhs dh[r,f] = sum_d dys[r,d] * wo[e,f,d] (the gradient
 * against the transposed wo), kept in fp32 and passed through the SwiGLU
 * backward when z is given (output dz [R,2F]), else stored as bf16 dh [R,F];
 * drhs dwo[e,f,d] = bf16(sum_{r in group e, ascending} h[r,f] * dys[r,d]),
 * zero for an empty group. */
int oracle_fc2_bwd(const uint16_t* dys, const uint16_t* h, const uint16_t* wo,
                   const uint16_t* z, const int32_t* offs, int E, int F, int D,
                   uint16_t* dh_or_dz, uint16_t* dwo) {
  if (E <= 0 || D <= 0 || F <= 0) return -1;
  const int R = offs[E];
  if (dh_or_dz) {
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < R; ++r) {
      int e = 0;
      while (offs[e + 1] <= r) ++e;
      const uint16_t* W = wo + (size_t)e * F * D;
      for (int f = 0; f < F; ++f) {
        float acc = 0.0f;
        for (int d = 0; d < D; ++d) acc = acc + BF(dys[(size_t)r * D + d]) * BF(W[(size_t)f * D + d]);
        if (z) {
          float dg, du;
          swiglu_bwd_one(acc, BF(z[(size_t)r * 2 * F + f]), BF(z[(size_t)r * 2 * F + F + f]), &dg, &du);
          dh_or_dz[(size_t)r * 2 * F + f] = RN(dg);
          dh_or_dz[(size_t)r * 2 * F + F + f] = RN(du);
        } else {
          dh_or_dz[(size_t)r * F + f] = RN(acc);
        }
      }
    }
  }
  if (dwo) {
#pragma omp parallel
    {
      float* a = (float*)malloc(sizeof(float) * (size_t)D);
#pragma omp for collapse(2) schedule(dynamic, 4)
      for (int e = 0; e < E; ++e)
        for (int f = 0; f < F; ++f) {
          for (int d = 0; d < D; ++d) a[d] = 0.0f;
          for (int r = offs[e]; r < offs[e + 1]; ++r) {
            float hv = BF(h[(size_t)r * F + f]);
            for (int d = 0; d < D; ++d) a[d] = a[d] + hv * BF(dys[(size_t)r * D + d]);
          }
          for (int d = 0; d < D; ++d) dwo[((size_t)e * F + f) * D + d] = RN(a[d]);
        }
      free(a);
    }
  }
  return 0;
}

/* The SwiGLU backward on its own, from a stored bf16 dh [R,F] and z [R,2F]. */
int oracle_swiglu_bwd(const uint16_t* dh, const uint16_t* z, int R, int F, uint16_t* dz) {
  if (R < 0 || F <= 0) return -1;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < R; ++r)
    for (int f = 0; f < F; ++f) {
      float dg, du;
      swiglu_bwd_one(BF(dh[(size_t)r * F + f]), BF(z[(size_t)r * 2 * F + f]),
                     BF(z[(size_t)r * 2 * F + F + f]), &dg, &du);
      dz[(size_t)r * 2 * F + f] = RN(dg);
      dz[(size_t)r * 2 * F + F + f] = RN(du);
    }
  return 0;
}

/* Backward of FC1 against the whole prefused wi: dlhs
 *   dxs[r,d] = bf16(sum_{n<2F} dz[r,n] * wi[e,d,n])  (the transposed wi),
 * drhs dwi[e,d,n] = bf16(sum_{r in group e, ascending} xs[r,d] * dz[r,n]),
 * zero for an empty group. */
int oracle_fc1_bwd(const uint16_t* dz, const uint16_t* xs, const uint16_t* wi,
                   const int32_t* offs, int E, int D, int F, uint16_t* dxs, uint16_t* dwi) {
  if (E <= 0 || D <= 0 || F <= 0) return -1;
  const int N = 2 * F;
  const int R = offs[E];
  if (dxs) {
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < R; ++r) {
      int e = 0;
      while (offs[e + 1] <= r) ++e;
      const uint16_t* W = wi + (size_t)e * D * N;
      for (int d = 0; d < D; ++d) {
        float acc = 0.0f;
        for (int n = 0; n < N; ++n) acc = acc + BF(dz[(size_t)r * N + n]) * BF(W[(size_t)d * N + n]);
        dxs[(size_t)r * D + d] = RN(acc);
      }
    }
  }
  if (dwi) {
#pragma omp parallel
    {
      float* a = (float*)malloc(sizeof(float) * (size_t)N);
#pragma omp for collapse(2) schedule(dynamic, 4)
      for (int e = 0; e < E; ++e)
        for (int d = 0; d < D; ++d) {
          for (int n = 0; n < N; ++n) a[n] = 0.0f;
          for (int r = offs[e]; r < offs[e + 1]; ++r) {
            float xv = BF(xs[(size_t)r * D + d]);
            for (int n = 0; n < N; ++n) a[n] = a[n] + xv * BF(dz[(size_t)r * N + n]);
          }
          for (int n = 0; n < N; ++n) dwi[((size_t)e * D + d) * N + n] = RN(a[n]);
        }
      free(a);
    }
  }
  return 0;
}

/* Backward of the permute [Fused p/c row 2]: the combine with unit weights,
 *   dx[t] = bf16(sum_{k ascending} dxs[pos[t,k]]). */
int oracle_permute_bwd(const uint16_t* dxs, const int32_t* pos, int T, int K, int D,
                       uint16_t* dx) {
  return oracle_combine(dxs, NULL, pos, T, K, D, dx);
}

/* ------------------------------------------------------------------ MXFP8
 * [TE MoE, Changes item 1 and Flowchart], with the format read as OCP MX
 * v1.0 MXFP8 (see oracle.h). */

/* E4M3 code -> value: sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent field 0 holds the subnormals m * 2^-9; S.1111.111 is NaN. */
double oracle_e4m3_to_f64(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

/* value -> E4M3 code, round to nearest with ties to even, magnitudes beyond
 * the largest finite value 448 saturated to it. */
uint8_t oracle_f64_to_e4m3(double v) {
  if (isnan(v)) return 0x7F;
  const uint8_t s = signbit(v) ? 0x80 : 0x00;
  const double a = fabs(v);
  if (a >= 448.0) return (uint8_t)(s | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal spacing 2^-9; rounding up to 8 * 2^-9 gives the smallest
     * normal, whose code is 8 as well */
    const double m = nearbyint(a * 512.0);
    return (uint8_t)(s | (uint8_t)m);
  }
  int ex;
  frexp(a, &ex);
  int E = ex - 1;                                /* a in [2^E, 2^(E+1)), E in [-6, 8] */
  double m = nearbyint(ldexp(a, 3 - E));         /* 8 .. 16: 1.mmm with 3 bits */
  if (m == 16.0) {
    m = 8.0;
    E += 1;
  }
  if (E > 8 || (E == 8 && m > 14.0)) return (uint8_t)(s | 0x7E);
  return (uint8_t)(s | (uint8_t)(((E + 7) << 3) | ((int)m - 8)));
}

/* Shared exponent of one block: floor(log2(amax)) - 8 (8 = the exponent of
 * E4M3's largest power of two), clamped below to E8M0's -127. */
static int mx_shared_exp(const float* v, int n) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) {
    const double a = fabs((double)v[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0) return -127;
  int ex;
  frexp(amax, &ex);
  const int s = (ex - 1) - 8;
  return s < -127 ? -127 : s;
}

int oracle_mx_quantize(const float* x, int rows, int K, uint8_t* q, uint8_t* sc) {
  if (rows < 0 || K <= 0 || K % 32 != 0) return -1;
  const int nb = K / 32;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < nb; ++b) {
      const float* v = x + (size_t)r * K + (size_t)b * 32;
      const int s = mx_shared_exp(v, 32);
      sc[(size_t)r * nb + b] = (uint8_t)(s + 127);
      for (int i = 0; i < 32; ++i)
        q[(size_t)r * K + (size_t)b * 32 + i] = oracle_f64_to_e4m3(ldexp((double)v[i], -s));
    }
  }
  return 0;
}

/* Dequantized row of n elements (n % 32 == 0): code * 2^(scale - 127). */
static void mx_row(const uint8_t* q, const uint8_t* sc, int n, double* out) {
  for (int i = 0; i < n; ++i) out[i] = ldexp(oracle_e4m3_to_f64(q[i]), (int)sc[i / 32] - 127);
}

/* FC1 + SwiGLU on MX operands: per row r of group e and output column n,
 * a[n] = sum_d x[r,d] * w[e,n,d] of the dequantized values (float64), then
 * h[r,f] = fp32(silu(a[f]) * a[F+f]). */
int oracle_mx_fc1_swiglu(const uint8_t* xq, const uint8_t* xsc, const uint8_t* wq,
                         const uint8_t* wsc, const int32_t* offs, int E, int D, int F,
                         float* h, uint16_t* z) {
  if (E <= 0 || D <= 0 || F <= 0 || D % 32 != 0) return -1;
  const int N = 2 * F, R = offs[E], nb = D / 32;
#pragma omp parallel
  {
    double* xr = (double*)malloc(sizeof(double) * (size_t)D);
    double* wr = (double*)malloc(sizeof(double) * (size_t)D);
    double* a = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 4)
    for (int r = 0; r < R; ++r) {
      int e = 0;
      while (offs[e + 1] <= r) ++e;
      mx_row(xq + (size_t)r * D, xsc + (size_t)r * nb, D, xr);
      for (int n = 0; n < N; ++n) {
        const size_t wrow = (size_t)e * N + n;
        mx_row(wq + wrow * D, wsc + wrow * nb, D, wr);
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += xr[d] * wr[d];
        a[n] = acc;
      }
      for (int f = 0; f < F; ++f) {
        const double g = a[f], u = a[F + f];
        h[(size_t)r * F + f] = (float)((g / (1.0 + exp(-g))) * u);
      }
      if (z)
        for (int n = 0; n < N; ++n) z[(size_t)r * N + n] = RN((float)a[n]);
    }
    free(xr);
    free(wr);
    free(a);
  }
  return 0;
}

/* FC2 on MX operands: ys[r,d] = bf16(fp32(sum_f h[r,f] * w[e,d,f])) of the
 * dequantized values (float64 sum). */
int oracle_mx_fc2(const uint8_t* hq, const uint8_t* hsc, const uint8_t* wq, const uint8_t* wsc,
                  const int32_t* offs, int E, int F, int D, uint16_t* ys) {
  if (E <= 0 || D <= 0 || F <= 0 || F % 32 != 0) return -1;
  const int R = offs[E], nb = F / 32;
#pragma omp parallel
  {
    double* hr = (double*)malloc(sizeof(double) * (size_t)F);
    double* wr = (double*)malloc(sizeof(double) * (size_t)F);
#pragma omp for schedule(dynamic, 4)
    for (int r = 0; r < R; ++r) {
      int e = 0;
      while (offs[e + 1] <= r) ++e;
      mx_row(hq + (size_t)r * F, hsc + (size_t)r * nb, F, hr);
      for (int d = 0; d < D; ++d) {
        const size_t wrow = (size_t)e * D + d;
        mx_row(wq + wrow * F, wsc + wrow * nb, F, wr);
        double acc = 0.0;
        for (int f = 0; f < F; ++f) acc += hr[f] * wr[f];
        ys[(size_t)r * D + d] = RN((float)acc);
      }
    }
    free(hr);
    free(wr);
  }
  return 0;
}

/* Elementwise RN of n fp32 values to bf16 bit patterns. */
int oracle_f32_to_bf16_array(const float* x, long n, uint16_t* out) {
  if (n < 0) return -1;
  for (long i = 0; i < n; ++i) out[i] = RN(x[i]);
  return 0;
}

/* ---------------------------------------------------------- MXFP8 backward
 * [TE MoE, Changes item 1: the block takes MXFP8 quantization in training;
 * Flowchart: the grouped GEMMs of the forward and of the backward].  Read
 * as: every GEMM of the backward takes both operands as MXFP8 with blocks
 * along its own contraction axis:
 *   FC2 dgrad  dh[r,f]    = sum_d dys[r,d] * wo[e,f,d]   dys along D, wo along its last axis;
 *   FC1 dgrad  dxs[r,d]   = sum_n dz[r,n] * wi[e,d,n]    dz along 2F, wi along its last axis
 *              (the form of oracle_mx_fc2 with wq = wi [E, D, 2F]);
 *   wgrads     dwo[e,f,d] = sum_{r in e} h[r,f] * dys[r,d],
 *              dwi[e,d,n] = sum_{r in e} xs[r,d] * dz[r,n]   both along the tokens of group e.
 * What is quantized is what the bf16 block keeps for its backward (xs, and
 * h and z rounded to bf16) and the bf16 gradients dys and dz. */

/* Token-axis quantization within groups: the rows of group e are cut into
 * blocks of 32 from its first row (its last block shorter); for each column
 * c the rows of one block share a scale, computed from those rows only (a
 * short block is as if padded with zeros).  x fp32 [R, C] -> q [R, C]
 * codes and sc [NB, C] scales, where block b of group e is scale row
 * boff[e] + b and boff[e] = sum_{e' < e} ceil(size_e' / 32) (boff [E+1] is
 * written; NB = boff[E]). */
int oracle_mx_quantize_tokens(const float* x, const int32_t* offs, int E, int C, uint8_t* q,
                              uint8_t* sc, int32_t* boff) {
  if (E <= 0 || C <= 0) return -1;
  boff[0] = 0;
  for (int e = 0; e < E; ++e) boff[e + 1] = boff[e] + (offs[e + 1] - offs[e] + 31) / 32;
  const int NB = boff[E];
#pragma omp parallel for schedule(dynamic, 4)
  for (int gb = 0; gb < NB; ++gb) {
    int e = 0;
    while (boff[e + 1] <= gb) ++e;
    const int r0 = offs[e] + 32 * (gb - boff[e]);
    const int n = offs[e + 1] - r0 < 32 ? offs[e + 1] - r0 : 32;
    float v[32];
    for (int c = 0; c < C; ++c) {
      for (int i = 0; i < n; ++i) v[i] = x[(size_t)(r0 + i) * C + c];
      const int s = mx_shared_exp(v, n);
      sc[(size_t)gb * C + c] = (uint8_t)(s + 127);
      for (int i = 0; i < n; ++i)
        q[(size_t)(r0 + i) * C + c] = oracle_f64_to_e4m3(ldexp((double)v[i], -s));
    }
  }
  return 0;
}

/* Weight gradient on operands quantized along tokens:
 *   out[e,i,j] = bf16(fp32(sum_{r in group e, ascending} A[r,i] * B[r,j]))
 * of the dequantized values (float64 sum), zero for an empty group.
 * A = (aq [R, Ca], asc [NB, Ca]) and B = (bq [R, Cb], bsc [NB, Cb]), both
 * from oracle_mx_quantize_tokens with these offsets (boff its output). */
int oracle_mx_wgrad(const uint8_t* aq, const uint8_t* asc, const uint8_t* bq, const uint8_t* bsc,
                    const int32_t* offs, const int32_t* boff, int E, int Ca, int Cb,
                    uint16_t* out) {
  if (E <= 0 || Ca <= 0 || Cb <= 0) return -1;
  double val[256], p2[256];
  for (int c = 0; c < 256; ++c) {
    val[c] = oracle_e4m3_to_f64((uint8_t)c);
    p2[c] = ldexp(1.0, c - 127);
  }
#pragma omp parallel
  {
    double* acc = (double*)malloc(sizeof(double) * (size_t)Cb);
#pragma omp for collapse(2) schedule(dynamic, 4)
    for (int e = 0; e < E; ++e)
      for (int i = 0; i < Ca; ++i) {
        for (int j = 0; j < Cb; ++j) acc[j] = 0.0;
        for (int r = offs[e]; r < offs[e + 1]; ++r) {
          const size_t blk = (size_t)boff[e] + (size_t)((r - offs[e]) / 32);
          const double a = val[aq[(size_t)r * Ca + i]] * p2[asc[blk * Ca + i]];
          for (int j = 0; j < Cb; ++j)
            acc[j] += a * (val[bq[(size_t)r * Cb + j]] * p2[bsc[blk * Cb + j]]);
        }
        for (int j = 0; j < Cb; ++j) out[((size_t)e * Ca + i) * Cb + j] = RN((float)acc[j]);
      }
    free(acc);
  }
  return 0;
}

/* FC2 dgrad with the SwiGLU backward on MX operands: per row r of group e,
 *   dh[r,f] = fp32(sum_d dys[r,d] * wo[e,f,d]) of the dequantized values
 * (float64 sum; dq/dsc = dys [R, D] with blocks along D, wq/wsc = wo
 * [E, F, D] with blocks along D), then dz[r,f], dz[r,F+f] =
 * bf16(swiglu_bwd(dh, z[r,f], z[r,F+f])) as in oracle_fc2_bwd. */
int oracle_mx_fc2_dgrad_swiglu(const uint8_t* dq, const uint8_t* dsc, const uint8_t* wq,
                               const uint8_t* wsc, const uint16_t* z, const int32_t* offs, int E,
                               int D, int F, uint16_t* dz) {
  if (E <= 0 || D <= 0 || F <= 0 || D % 32 != 0) return -1;
  const int R = offs[E], nb = D / 32;
#pragma omp parallel
  {
    double* dr = (double*)malloc(sizeof(double) * (size_t)D);
    double* wr = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
    for (int r = 0; r < R; ++r) {
      int e = 0;
      while (offs[e + 1] <= r) ++e;
      mx_row(dq + (size_t)r * D, dsc + (size_t)r * nb, D, dr);
      for (int f = 0; f < F; ++f) {
        const size_t wrow = (size_t)e * F + f;
        mx_row(wq + wrow * D, wsc + wrow * nb, D, wr);
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += dr[d] * wr[d];
        float dg, du;
        swiglu_bwd_one((float)acc, BF(z[(size_t)r * 2 * F + f]), BF(z[(size_t)r * 2 * F + F + f]),
                       &dg, &du);
        dz[(size_t)r * 2 * F + f] = RN(dg);
        dz[(size_t)r * 2 * F + F + f] = RN(du);
      }
    }
    free(dr);
    free(wr);
  }
  return 0;
}
