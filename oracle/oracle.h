/*
 * CPU oracle for the sparse MoE expert block -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the package's smoke check and the benchmark's
 * CPU-baseline leg may load this library.  The CUDA path never links,
 * includes or calls it, and it shares no code with the CUDA path.
 *
 * Conventions (shared with the CUDA path only through the statement of the
 * problem, never through code):
 *   T tokens, D = emb, E experts, K = top_k, F = mlp, R = T*K.
 *   bf16 tensors are passed as raw uint16 bit patterns, row-major.
 *   Every float sum is accumulated in fp32 from 0.0f in ascending index
 *   order; bf16 rounding (round-to-nearest-even) happens exactly where a
 *   tensor is stored.  Compiled with -ffp-contract=off so that no multiply
 *   and add are fused.
 *
 * Every function returns 0 on success, a negative value on bad arguments,
 * and (routing/histogram only) a positive count of expert ids outside [0,E).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_SOFTMAX_TOPK = 0, ORACLE_SIGMOID_NORM = 1, ORACLE_GIVEN = 2 };

/* f32 -> bf16 round-to-nearest-even and bf16 -> f32, exposed for tests. */
uint16_t oracle_f32_to_bf16(float f);
float oracle_bf16_to_f32(uint16_t b);

int oracle_route(const float* logits, const float* bias, int mode,
                 int T, int E, int K, int32_t* ids, float* w);
int oracle_histogram(const int32_t* ids, int T, int K, int E,
                     int32_t* group_sizes, int32_t* group_offsets,
                     int32_t* pos, int32_t* row_src);
int oracle_permute(const uint16_t* x, const int32_t* pos, int T, int K, int D,
                   uint16_t* xs);
int oracle_fc1_swiglu(const uint16_t* xs, const uint16_t* wi,
                      const int32_t* group_offsets, int E, int D, int F,
                      uint16_t* h, uint16_t* z);
int oracle_fc2(const uint16_t* h, const uint16_t* wo, const int32_t* group_offsets,
               int E, int F, int D, uint16_t* ys);
int oracle_combine(const uint16_t* ys, const float* w, const int32_t* pos,
                   int T, int K, int D, uint16_t* out);
int oracle_combine_bwd(const uint16_t* dout, const uint16_t* ys, const float* w,
                       const int32_t* pos, int T, int K, int D,
                       uint16_t* dys, float* dw);
int oracle_fc2_bwd(const uint16_t* dys, const uint16_t* h, const uint16_t* wo,
                   const uint16_t* z, const int32_t* group_offsets,
                   int E, int F, int D, uint16_t* dh_or_dz, uint16_t* dwo);
int oracle_swiglu_bwd(const uint16_t* dh, const uint16_t* z, int R, int F,
                      uint16_t* dz);
int oracle_fc1_bwd(const uint16_t* dz, const uint16_t* xs, const uint16_t* wi,
                   const int32_t* group_offsets, int E, int D, int F,
                   uint16_t* dxs, uint16_t* dwi);
int oracle_permute_bwd(const uint16_t* dxs, const int32_t* pos, int T, int K, int D,
                       uint16_t* dx);
int oracle_num_threads(void);

/*
 * MXFP8 forward [TE MoE, Changes item 1 ("MXFP8 quantization in the MoE
 * block") and Flowchart ("Grouped FC1 quantize and GEMM" -> "Activation and
 * grouped FC2 GEMM")].  The pages name the format only; its definition is
 * read as the OCP Microscaling (MX) v1.0 MXFP8 format: blocks of 32
 * consecutive elements along the contraction axis share one E8M0 scale
 * (the byte c means 2^(c-127)); each element is an E4M3 code (bias 7, no
 * infinities, S.1111.111 = NaN, largest finite 448).
 *   Block quantization: X = 2^s, s = max(floor(log2(amax)) - 8, -127)
 *   (s = -127 when amax = 0), code_i = E4M3(v_i / X) rounded to nearest,
 *   ties to even, magnitudes beyond 448 saturated to 448.
 * The MX GEMMs sum the exact products of dequantized elements in float64 in
 * ascending index order (nothing but the sum's rounding differs from the
 * real-number result).
 */
double oracle_e4m3_to_f64(uint8_t c);
uint8_t oracle_f64_to_e4m3(double v);
/* x fp32 [rows, K], K % 32 == 0 -> q [rows, K] codes, sc [rows, K/32]. */
int oracle_mx_quantize(const float* x, int rows, int K, uint8_t* q, uint8_t* sc);
/* FC1 + SwiGLU on MX operands: xq/xsc [R, D] / [R, D/32]; wq/wsc are wi
 * transposed, [E, 2F, D] / [E, 2F, D/32] (row n = output column n; gate =
 * rows [0,F), up = [F,2F)).  h fp32 [R, F] = fp32(silu(g) * u) of the
 * float64 sums. */
int oracle_mx_fc1_swiglu(const uint8_t* xq, const uint8_t* xsc, const uint8_t* wq,
                         const uint8_t* wsc, const int32_t* group_offsets, int E, int D, int F,
                         float* h);
/* FC2 on MX operands: hq/hsc [R, F] / [R, F/32]; wq/wsc are wo transposed,
 * [E, D, F] / [E, D, F/32].  ys bf16 [R, D] = bf16(fp32(sum)). */
int oracle_mx_fc2(const uint8_t* hq, const uint8_t* hsc, const uint8_t* wq, const uint8_t* wsc,
                  const int32_t* group_offsets, int E, int F, int D, uint16_t* ys);

#ifdef __cplusplus
}
#endif
#endif
