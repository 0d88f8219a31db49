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
 * float64 sums; z (may be NULL) bf16 [R, 2F] = bf16(fp32(sum)) of every
 * output column, kept for the backward. */
int oracle_mx_fc1_swiglu(const uint8_t* xq, const uint8_t* xsc, const uint8_t* wq,
                         const uint8_t* wsc, const int32_t* group_offsets, int E, int D, int F,
                         float* h, uint16_t* z);
/* FC2 on MX operands: hq/hsc [R, F] / [R, F/32]; wq/wsc are wo transposed,
 * [E, D, F] / [E, D, F/32].  ys bf16 [R, D] = bf16(fp32(sum)). */
int oracle_mx_fc2(const uint8_t* hq, const uint8_t* hsc, const uint8_t* wq, const uint8_t* wsc,
                  const int32_t* group_offsets, int E, int F, int D, uint16_t* ys);
int oracle_f32_to_bf16_array(const float* x, long n, uint16_t* out);

/*
 * MXFP8 backward [TE MoE, Changes item 1; Flowchart].  Every GEMM of the
 * backward on MX operands with blocks along its own contraction axis: the
 * dgrads take the gradient rows (blocks along the row) and the weight
 * quantized along its last axis; the wgrads take both operands quantized
 * along the tokens of each group, in blocks of 32 rows from the group's
 * first row (a group's last block may be short).  The quantized tensors are
 * the bf16 ones the block keeps (xs, h, z) and the bf16 gradients.
 */
/* x fp32 [R, C] -> q [R, C], sc [NB, C], boff [E+1]: block b of group e
 * covers rows offs[e] + 32b .. min(offs[e] + 32b + 32, offs[e+1]) and its
 * scales are row boff[e] + b of sc, boff[e] = sum_{e'<e} ceil(size_e'/32). */
int oracle_mx_quantize_tokens(const float* x, const int32_t* group_offsets, int E, int C,
                              uint8_t* q, uint8_t* sc, int32_t* boff);
/* out bf16 [E, Ca, Cb] = bf16(fp32(sum_{r in group e} A[r,i] * B[r,j])) on
 * token-quantized A [R, Ca] and B [R, Cb]; zero for an empty group. */
int oracle_mx_wgrad(const uint8_t* aq, const uint8_t* asc, const uint8_t* bq, const uint8_t* bsc,
                    const int32_t* group_offsets, const int32_t* boff, int E, int Ca, int Cb,
                    uint16_t* out);
/* dz bf16 [R, 2F] = SwiGLU backward of dh = fp32(sum_d dys[r,d] * wo[e,f,d])
 * (dys [R, D] and wo [E, F, D] both with blocks along D) at z bf16 [R, 2F]. */
int oracle_mx_fc2_dgrad_swiglu(const uint8_t* dq, const uint8_t* dsc, const uint8_t* wq,
                               const uint8_t* wsc, const uint16_t* z,
                               const int32_t* group_offsets, int E, int D, int F, uint16_t* dz);

#ifdef __cplusplus
}
#endif
#endif
