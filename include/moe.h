/*
 * moe.h -- C ABI of libmoe.so, the single-GPU sparse mixture-of-experts
 * expert block for NVIDIA GB300 (sm_103a).
 *
 * The block (forward):
 *   route    -> top-k expert ids and routing weights per token
 *   histogram-> group_size per expert, expert-sorted position of every slot
 *   permute  -> xs: tokens gathered into expert-sorted order
 *   FC1      -> one grouped GEMM against the whole prefused wi [E, emb, 2*mlp],
 *               SwiGLU applied to its output activations
 *   FC2      -> grouped GEMM against wo [E, mlp, emb]
 *   combine  -> unpermute plus the top-k weighted sum
 * and the backward of every step.
 *
 * Sources the operations follow (pages of the MoE optimisation discussions):
 *   [Keep fused]  MaxText "Keep fused MoE weights intact through FSDP gather",
 *                 Description: the prefused [experts, embed, 2*mlp] weight goes
 *                 through one grouped GEMM; only its output is split into gate
 *                 and up activations for SwiGLU.
 *   [Fused p/c]   MaxText "MoE: fused TensorCore Pallas permute/combine kernels
 *                 and split-expert wi layout for TPU v6e", Context item 1 and
 *                 Commits table rows 1-2: the permute gathers tokens into
 *                 expert-sorted order without an unsorted [tokens*top_k, emb]
 *                 copy, with the group_size histogram computed first; its
 *                 backward is the combine with unit weights; the combine is the
 *                 unpermute plus the top-K weighted sum, whose backward is a
 *                 permutation for dx and a per-slot reduction for dw.
 *   [Gemma4 L/M]  MaxText "Gemma4 26B MoE on TPU v6e: MaxText layer/model
 *                 optimizations", Commits table row 6 (top_k_weights and
 *                 group_size) and row 7 (gate/up split backward = one
 *                 concatenation).
 *   [TE MoE]      TransformerEngine "[DRAFT][JAX] Optimize MoE block", Changes
 *                 (group-aware grouped GEMM, no masking pass) and Flowchart.
 *   [Transposed]  The "transposed-RHS gmm_v2 kernel for the backward dlhs"
 *                 named under Related PRs of [Fused p/c]: dlhs multiplies by
 *                 the transposed expert weight.
 *
 * Notation: T tokens, D = emb, E experts, K = top_k, F = mlp, R = T*K.
 * All tensors are dense, row-major, and live in DEVICE memory owned by the
 * caller (for example PyTorch tensors).  bf16 tensors are raw IEEE bfloat16
 * bit patterns (moe_bf16).  The library never allocates device memory:
 * scratch comes from `ws`, at least moe_workspace_bytes(d) bytes.
 *
 * Every call is asynchronous and stream-ordered on `stream`; none blocks the
 * host or reads group sizes back to it.  Host-side argument errors are
 * returned synchronously before anything is enqueued:
 *   MOE_ERR_INVALID_ARG  a required pointer is NULL or not 16-byte aligned;
 *   MOE_ERR_UNSUPPORTED  D % 64 != 0, F % 64 != 0, K < 1, K > E, K > 32,
 *                        E > 1024, T < 0, or R >= 2^31;
 *   MOE_ERR_CUDA         a kernel launch failed (cudaGetLastError).
 * Errors found on the device are written to *dev_status (an int32 in device
 * memory that the caller zeroes and reads after synchronising; the first
 * error wins):
 *   MOE_ERR_DEVICE       an expert id outside [0, E) (its slot is dropped:
 *                        pos = -1, not counted in group_sizes);
 *   MOE_ERR_TIMEOUT      a bounded wait inside a kernel gave up (the kernel
 *                        released its resources and returned).
 * T = 0 is valid: the calls do nothing but zero group_sizes/group_offsets.
 * Gradient outputs overwrite their buffers; they never accumulate.
 * The functions keep no state between calls apart from a per-device cache of
 * the SM count and of a driver entry point, and are safe to call from several
 * host threads; calls that share a `ws` must be ordered on one stream.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_CUDA = 3,
  MOE_ERR_DEVICE = 4,
  MOE_ERR_TIMEOUT = 5
} moe_status;

typedef struct {
  int32_t T; /* tokens */
  int32_t D; /* emb, multiple of 64 */
  int32_t E; /* experts, 1..1024 */
  int32_t K; /* top_k, 1..min(E, 32) */
  int32_t F; /* mlp, multiple of 64 */
} moe_dims;

typedef enum {
  MOE_SCORE_SOFTMAX_TOPK = 0, /* w = softmax over the K selected scores */
  MOE_SCORE_SIGMOID_NORM = 1, /* w = sigmoid(selected) / sum of the K sigmoids */
  MOE_SCORE_GIVEN = 2         /* ids and w are inputs; only the histogram runs */
} moe_score_mode;

typedef uint16_t moe_bf16; /* raw bfloat16 bits */

/* Bytes of scratch that every call below may use through `ws` for dims d
 * (the largest need over all calls). */
size_t moe_workspace_bytes(moe_dims d);

/* A static English description of a status code. */
const char* moe_status_string(moe_status s);

/* Version of this ABI; lets a loader check the library it opened without
 * touching a GPU.  2: adds the MXFP8 entry points (moe_mx_*) and the FC1
 * calls over expert ranges (moe_grouped_gemm_fc1_*_experts) to version 1's.
 * 3: adds moe_fused_forward.  4: adds the MXFP8 backward
 * (moe_mx_grouped_gemm_fc2_bwd and _fc1_bwd, moe_mx_quantize_rows, moe_mx_quantize_tokens, the backward's MX buffers),
 * z to moe_mx_grouped_gemm_fc1_swiglu and the dgrad copies to
 * moe_mx_quantize_wi/wo. */
int moe_abi_version(void);

/*
 * Routing and group_size histogram [Gemma4 L/M row 6; Fused p/c row 2].
 *   logits  fp32 [T,E]   router logits (ignored, may be NULL, for GIVEN)
 *   bias    fp32 [E]     per-expert bias added to the logits, or NULL
 *   mode    score mode: the score of expert e is s = logit + bias[e]; the K
 *           largest scores are taken in descending order (equal scores: the
 *           lower expert id first) and weighted by `mode`
 *   ids     int32 [T,K]  out (in for GIVEN): expert id of slot (t,k)
 *   w       fp32 [T,K]   out (in for GIVEN, may then be NULL): routing weight
 *   group_sizes   int32 [E]    out: rows routed to each expert
 *   group_offsets int32 [E+1]  out: exclusive prefix sum of group_sizes
 *   pos     int32 [T,K]  out: expert-sorted row of slot (t,k); the order is
 *           stable in the flat slot index j = t*K + k
 *   row_src int32 [R]    out: row_src[pos[j]] = j (rows never filled: -1)
 *   dev_status int32*    device error word (may be NULL)
 *   ws      scratch, moe_workspace_bytes(d) bytes
 */
moe_status moe_route_histogram(const float* logits, const float* bias, moe_score_mode mode,
                               int32_t* ids, float* w, int32_t* group_sizes,
                               int32_t* group_offsets, int32_t* pos, int32_t* row_src,
                               int32_t* dev_status, void* ws, moe_dims d, cudaStream_t stream);

/*
 * moe_route_histogram without a workspace argument.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory,
 * such as code running inside another framework's operator or plugin that
 * is handed only the buffers its planner sized, or latency-critical code
 * that must not call cudaMalloc (it can synchronise the device).  It
 * computes exactly what moe_route_histogram computes, from the same
 * arguments minus `ws`, and allocates nothing: its scratch (the per-chunk
 * expert counts and their prefixes) is a fixed array of 262144 int32
 * (1 MiB) inside the library, held by every GPU that loads the library
 * until the process exits.
 *   Limit: 2 * ceil(T/256) * E <= 262144 (e.g. T = 32768 with E <= 1024);
 *   larger dims return MOE_ERR_UNSUPPORTED without launching anything.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is cached per device together
 *   with the id of the device's CUDA context; a call in a new context (for
 *   example after cudaDeviceReset) looks it up again, so that call too must
 *   come before any capture.
 *   All calls share the one array: each call clears the counts it uses and
 *   rewrites the prefixes it reads, so earlier calls leave nothing behind,
 *   but calls that overlap on the GPU (different streams, or several host
 *   threads) race on it and must be ordered by the caller.
 */
moe_status moe_route_histogram_noalloc(const float* logits, const float* bias, moe_score_mode mode,
                                       int32_t* ids, float* w, int32_t* group_sizes,
                                       int32_t* group_offsets, int32_t* pos, int32_t* row_src,
                                       int32_t* dev_status, moe_dims d, cudaStream_t stream);

/*
 * Permute [Fused p/c Context item 1, row 2]: xs[pos[t,k]] = x[t] for every
 * slot with pos >= 0 (an exact copy; each x row is read once and written K
 * times; no unsorted [R, D] copy exists).
 *   x  bf16 [T,D] in;  pos int32 [T,K] in;  xs bf16 [R,D] out.
 */
moe_status moe_permute(const moe_bf16* x, const int32_t* pos, moe_bf16* xs, moe_dims d,
                       cudaStream_t stream);

/*
 * Permute backward [Fused p/c row 2] = the combine with unit weights:
 *   dx[t] = bf16(sum_{k ascending} dxs[pos[t,k]])  (fp32 sum).
 *   dxs bf16 [R,D] in;  pos int32 [T,K] in;  dx bf16 [T,D] out.
 */
moe_status moe_permute_bwd(const moe_bf16* dxs, const int32_t* pos, moe_bf16* dx, moe_dims d,
                           cudaStream_t stream);

/*
 * FC1 + SwiGLU [Keep fused, Description; TE MoE, Changes and Flowchart]:
 * for every row r of group e (rows group_offsets[e] .. group_offsets[e+1]-1)
 *   a = xs[r] . wi[e]   (fp32 accumulation, N = 2F columns, wi never split)
 *   h[r,f] = bf16(silu(a[f]) * a[F+f]),  z[r,:] = bf16(a)  (when z != NULL)
 * Gate = columns [0,F) of wi's last axis, up = [F,2F).
 *   xs bf16 [R,D];  wi bf16 [E,D,2F];  group_offsets int32 [E+1] (device);
 *   h bf16 [R,F] out;  z bf16 [R,2F] out or NULL (inference).
 * Rows at or beyond group_offsets[E] are neither read nor written.
 */
moe_status moe_grouped_gemm_fc1_swiglu(const moe_bf16* xs, const moe_bf16* wi,
                                       const int32_t* group_offsets, moe_bf16* h, moe_bf16* z,
                                       int32_t* dev_status, void* ws, moe_dims d,
                                       cudaStream_t stream);

/*
 * FC1 backward against the whole wi [Transposed; TE MoE]:
 *   dlhs: dxs[r,d] = bf16(sum_{n<2F} dz[r,n] * wi[e,d,n])
 *   drhs: dwi[e,d,n] = bf16(sum_{r in group e} xs[r,d] * dz[r,n]); zero for
 *         an empty group.
 * grad is dz bf16 [R,2F] when z == NULL.  When z != NULL, grad is dh bf16
 * [R,F] and the SwiGLU backward [Gemma4 L/M row 7] runs first, writing
 * dz = [dgate | dup] into ws.  dxs (bf16 [R,D]) or dwi (bf16 [E,D,2F]) may be
 * NULL to skip that half.  ws is required when z != NULL or dwi != NULL (the
 * drhs keeps the counter of its dynamic tile schedule in the first bytes of
 * ws and resets it itself; ws needs no initial contents).
 */
moe_status moe_grouped_gemm_fc1_swiglu_bwd(const moe_bf16* grad, const moe_bf16* z,
                                           const moe_bf16* xs, const moe_bf16* wi,
                                           const int32_t* group_offsets, moe_bf16* dxs,
                                           moe_bf16* dwi, int32_t* dev_status, void* ws,
                                           moe_dims d, cudaStream_t stream);

/*
 * FC1 for one range of experts whose weights are a separate buffer: the
 * split-expert wi layout [Fused p/c, Context item 2 and Commits table row 3]
 * stores wi as expert halves that are gathered separately and consumed by
 * two chained grouped GEMM calls writing into one shared output buffer.
 * Here any split works: a call covers experts [e_begin, e_end) with
 * wi_part = their [e_end - e_begin, D, 2F] weights, and computes exactly
 * the rows moe_grouped_gemm_fc1_swiglu computes for those groups (rows
 * group_offsets[e_begin] .. group_offsets[e_end]-1 of h, and of z when
 * given); other rows are untouched.  Calls over ranges that tile [0, E)
 * give the whole FC1.  0 <= e_begin < e_end <= E, else MOE_ERR_INVALID_ARG.
 */
moe_status moe_grouped_gemm_fc1_swiglu_experts(const moe_bf16* xs, const moe_bf16* wi_part,
                                               const int32_t* group_offsets, int32_t e_begin,
                                               int32_t e_end, moe_bf16* h, moe_bf16* z,
                                               int32_t* dev_status, void* ws, moe_dims d,
                                               cudaStream_t stream);

/*
 * The FC1 backward for one range of experts (see above): from dz bf16
 * [R,2F], dlhs writes the rows of groups [e_begin, e_end) of dxs against
 * wi_part, and drhs writes dwi_part [e_end - e_begin, D, 2F] (zero for an
 * empty group).  Either output may be NULL, not both; ws is required with
 * dwi_part (the counter of the drhs's dynamic tile schedule).
 */
moe_status moe_grouped_gemm_fc1_bwd_experts(const moe_bf16* dz, const moe_bf16* xs,
                                            const moe_bf16* wi_part,
                                            const int32_t* group_offsets, int32_t e_begin,
                                            int32_t e_end, moe_bf16* dxs, moe_bf16* dwi_part,
                                            int32_t* dev_status, void* ws, moe_dims d,
                                            cudaStream_t stream);

/*
 * FC2 [TE MoE, Flowchart "grouped FC2 GEMM"]:
 *   ys[r,:] = bf16(h[r] . wo[e])  (fp32 accumulation).
 *   h bf16 [R,F];  wo bf16 [E,F,D];  ys bf16 [R,D] out.
 */
moe_status moe_grouped_gemm_fc2(const moe_bf16* h, const moe_bf16* wo,
                                const int32_t* group_offsets, moe_bf16* ys,
                                int32_t* dev_status, void* ws, moe_dims d, cudaStream_t stream);

/*
 * FC2 backward [Transposed; Gemma4 L/M row 7]:
 *   dlhs: dh[r,f] = sum_d dys[r,d] * wo[e,f,d] in fp32; with z != NULL the
 *         SwiGLU backward is fused on that fp32 value (s = sigmoid(g),
 *         g = z[r,f], u = z[r,F+f]):
 *           dz[r,f]   = bf16(dh * u * s * (1 + g*(1-s)))
 *           dz[r,F+f] = bf16(dh * g * s)
 *         and dh_or_dz is dz bf16 [R,2F]; with z == NULL it is dh bf16 [R,F].
 *   drhs: dwo[e,f,d] = bf16(sum_{r in group e} h[r,f] * dys[r,d]); zero for
 *         an empty group.
 * dh_or_dz or dwo may be NULL to skip that half.  ws is required when dwo !=
 * NULL (the counter of the drhs's dynamic tile schedule; no initial contents
 * needed).
 */
moe_status moe_grouped_gemm_fc2_bwd(const moe_bf16* dys, const moe_bf16* h, const moe_bf16* wo,
                                    const moe_bf16* z, const int32_t* group_offsets,
                                    moe_bf16* dh_or_dz, moe_bf16* dwo, int32_t* dev_status,
                                    void* ws, moe_dims d, cudaStream_t stream);

/*
 * Combine [Fused p/c row 1]: unpermute plus the top-K weighted sum,
 *   out[t] = bf16(sum_{k ascending} w[t,k] * ys[pos[t,k]])  (fp32, each
 *   product and sum rounded separately, slots with pos < 0 skipped).
 *   ys bf16 [R,D];  w fp32 [T,K];  pos int32 [T,K];  out bf16 [T,D].
 */
moe_status moe_combine(const moe_bf16* ys, const float* w, const int32_t* pos, moe_bf16* out,
                       moe_dims d, cudaStream_t stream);

/*
 * Combine backward [Fused p/c row 1]: a permutation for the activation
 * gradient and a per-slot reduction for the routing-weight gradient,
 *   dys[pos[t,k]] = bf16(w[t,k] * dout[t])
 *   dw[t,k] = sum_d dout[t,d] * ys[pos[t,k],d]  (fp32; 0 when pos < 0)
 *   dout bf16 [T,D];  ys bf16 [R,D];  w fp32 [T,K];  pos int32 [T,K];
 *   dys bf16 [R,D] out;  dw fp32 [T,K] out.
 */
moe_status moe_combine_bwd(const moe_bf16* dout, const moe_bf16* ys, const float* w,
                           const int32_t* pos, moe_bf16* dys, float* dw, moe_dims d,
                           cudaStream_t stream);

/*
 * ------------------------------------------------------------------ MXFP8
 * The forward in MXFP8 [TE MoE, Changes item 1 ("MXFP8 quantization in the
 * MoE block") and Flowchart ("Grouped FC1 quantize and GEMM" -> "Activation
 * and grouped FC2 GEMM")].  MXFP8 is read as the OCP MX v1.0 format: each
 * block of 32 consecutive elements along a GEMM's contraction axis shares
 * one E8M0 scale byte c (value 2^(c-127)); each element is an E4M3 code
 * (bias 7, no infinities, largest finite 448).  Quantizing a block:
 *   s = max(floor(log2(amax)) - 8, -127)  (s = -127 when amax = 0),
 *   c = s + 127,  code_i = E4M3(v_i * 2^-s), nearest-even, saturating.
 * Inputs must be finite.
 *
 * Scale blocks.  Scales are stored in 512-byte blocks, each covering 128
 * rows and one k-block of 128 contraction elements (4 scales per row): the
 * scale of row m (0..127) for elements [32j, 32j+32) of the k-block is byte
 * (m % 32) * 16 + (m / 32) * 4 + j, the order the tensor cores read.
 * KB(k) = ceil(k / 128) k-blocks; bytes of a block past the contraction
 * length, or for rows past the tensor's rows, are never used.
 *
 * Activation layout (xq/xsc, hq/hsc; rows in expert-sorted order): codes
 * [R, k] row-major.  Scales are tile-blocked: the rows of each group e are
 * cut into 128-row tiles starting at group_offsets[e]; the tiles of all
 * groups are numbered in order (group e's first tile is
 * tb[e] = sum_{e' < e} ceil(group_size[e'] / 128)), and tile g's scales
 * for k-block kb are the block at byte (g * KB(k) + kb) * 512.
 *
 * Weight layout (wq/wsc): the weight transposed so that its contraction
 * axis is contiguous, codes [E, N, k] (FC1: N = 2F rows, k = D; FC2: N = D,
 * k = F), scales [E, KB(k), NBp, 512] with NBp = 2 * ceil(N / 256) blocks
 * of 128 rows.  FC1's rows are interleaved in 64-row chunks, gate then up:
 * column n of wi (gate f = n for n < F, up f = n - F) is row
 * 128 * (f / 64) + 64 * (n >= F) + f % 64.
 *
 * moe_mx_bytes(d, which) gives each buffer's size in bytes.
 */
typedef enum {
  MOE_MX_XQ = 0,   /* xq codes [R, D] */
  MOE_MX_XSC = 1,  /* xq scales, tile-blocked, (ceil(R/128) + E) * KB(D) * 512 */
  MOE_MX_WIQ = 2,  /* wi codes [E, 2F, D] */
  MOE_MX_WISC = 3, /* wi scales [E, KB(D), 2*ceil(2F/256), 512] */
  MOE_MX_WOQ = 4,  /* wo codes [E, D, F] */
  MOE_MX_WOSC = 5, /* wo scales [E, KB(F), 2*ceil(D/256), 512] */
  MOE_MX_HQ = 6,   /* hq codes [R, F] */
  MOE_MX_HSC = 7,  /* hq scales, tile-blocked, (ceil(R/128) + E) * KB(F) * 512 */
  /* backward (see the MXFP8 backward below) */
  MOE_MX_DYQ = 8,        /* dys codes [R, D], blocks along D */
  MOE_MX_DYSC = 9,       /* their scales, tile-blocked, TB * KB(D) * 512 */
  MOE_MX_DZQ = 10,       /* dz codes [R, 2F], blocks along 2F */
  MOE_MX_DZSC = 11,      /* tile-blocked, TB * KB(2F) * 512 */
  MOE_MX_WIQ_BWD = 12,   /* wi codes [E, D, 2F], blocks along 2F */
  MOE_MX_WISC_BWD = 13,  /* [E, KB(2F), 2*ceil(D/256), 512] */
  MOE_MX_WOQ_BWD = 14,   /* wo codes [E, F, D], blocks along D */
  MOE_MX_WOSC_BWD = 15,  /* [E, KB(D), 2*ceil(F/256), 512] */
  MOE_MX_XT = 16,        /* xs along tokens: codes [D, Rp] */
  MOE_MX_XTSC = 17,      /* [TB, 2*ceil(D/256), 512] */
  MOE_MX_HT = 18,        /* h along tokens: codes [F, Rp] */
  MOE_MX_HTSC = 19,      /* [TB, 2*ceil(F/256), 512] */
  MOE_MX_DYT = 20,       /* dys along tokens: codes [D, Rp] */
  MOE_MX_DYTSC = 21,     /* [TB, 2*ceil(D/256), 512] */
  MOE_MX_DZT = 22,       /* dz along tokens: codes [2F, Rp] */
  MOE_MX_DZTSC = 23      /* [TB, 2*ceil(2F/256), 512] */
} moe_mx_buffer;

/* Bytes of MX buffer `which` for dims d (0 for invalid dims or `which`). */
size_t moe_mx_bytes(moe_dims d, moe_mx_buffer which);

/*
 * Grouped quantize of the expert weights (once per weight update), one read
 * of the weight for both of its MX copies:
 *   moe_mx_quantize_wi: wi bf16 [E, D, 2F] -> wq [E, 2F, D] (interleaved
 *                       rows) + wsc, blocks along D (the forward's FC1), and
 *                       wq_bwd [E, D, 2F] + wsc_bwd, blocks along 2F (the
 *                       FC1 dgrad; see the MXFP8 backward below);
 *   moe_mx_quantize_wo: wo bf16 [E, F, D]  -> wq [E, D, F] + wsc, blocks
 *                       along F (FC2), and wq_bwd [E, F, D] + wsc_bwd,
 *                       blocks along D (the FC2 dgrad).
 * Each (codes, scales) pair may be NULL (both of it), not both pairs.
 * Scale bytes of padding blocks are left as they are.
 */
moe_status moe_mx_quantize_wi(const moe_bf16* wi, uint8_t* wq, uint8_t* wsc, uint8_t* wq_bwd,
                              uint8_t* wsc_bwd, moe_dims d, cudaStream_t stream);
moe_status moe_mx_quantize_wo(const moe_bf16* wo, uint8_t* wq, uint8_t* wsc, uint8_t* wq_bwd,
                              uint8_t* wsc_bwd, moe_dims d, cudaStream_t stream);

/*
 * Grouped FC1 quantize [TE MoE, Flowchart]: the permute of moe_permute with
 * each token row quantized once (blocks along D) and its codes written to
 * xq[pos[t,k]] for every slot with pos >= 0; the scales go to the
 * tile-blocked xsc of the destination row.  Needs the group_offsets of the
 * histogram that produced pos.
 *   x bf16 [T,D];  pos int32 [T,K];  group_offsets int32 [E+1];
 *   xq [R,D] out;  xsc out.
 */
moe_status moe_mx_permute_quantize(const moe_bf16* x, const int32_t* pos,
                                   const int32_t* group_offsets, uint8_t* xq, uint8_t* xsc,
                                   moe_dims d, cudaStream_t stream);

/*
 * FC1 + SwiGLU on MX operands: for every row r of group e
 *   a[n] = sum_d x[r,d] * wi[e,d,n] of the dequantized operands (fp32
 *   accumulation of exact products), g = a[:F], u = a[F:],
 *   h[r,f] = fp32(silu(g_f) * u_f), written as MX codes hq [R,F] with the
 *   tile-blocked scales hsc (blocks along F: the A operand of the MX FC2)
 *   and/or as bf16 h [R,F].  hq/hsc (both or neither) and h may each be
 *   NULL, not all three.  z (may be NULL) bf16 [R, 2F] = bf16(a) in wi's
 *   column order [gate | up], kept for the backward.
 */
moe_status moe_mx_grouped_gemm_fc1_swiglu(const uint8_t* xq, const uint8_t* xsc,
                                          const uint8_t* wq, const uint8_t* wsc,
                                          const int32_t* group_offsets, uint8_t* hq,
                                          uint8_t* hsc, moe_bf16* h, moe_bf16* z,
                                          int32_t* dev_status, moe_dims d, cudaStream_t stream);

/*
 * FC2 on MX operands: ys[r,:] = bf16(sum_f h[r,f] * wo[e,f,:]) of the
 * dequantized operands (fp32 accumulation).
 *   hq, hsc from moe_mx_grouped_gemm_fc1_swiglu;  wq, wsc from
 *   moe_mx_quantize_wo;  ys bf16 [R,D] out.
 */
moe_status moe_mx_grouped_gemm_fc2(const uint8_t* hq, const uint8_t* hsc, const uint8_t* wq,
                                   const uint8_t* wsc, const int32_t* group_offsets,
                                   moe_bf16* ys, int32_t* dev_status, moe_dims d,
                                   cudaStream_t stream);

/*
 * MXFP8 backward [TE MoE, Changes item 1: MXFP8 quantization in the MoE
 * block, which trains; Flowchart].  Every backward GEMM takes both operands
 * as MXFP8 with blocks along its own contraction axis (format and scale
 * blocks as above):
 *   FC2 dgrad  dh[r,f] = sum_d dys[r,d] * wo[e,f,d]: dys quantized along D
 *              (moe_mx_quantize_rows), wo along its last axis
 *              (wq_bwd of moe_mx_quantize_wo); dh (fp32) goes straight into the
 *              SwiGLU backward at z, giving dz bf16 [R, 2F] = [dgate | dup];
 *   FC1 dgrad  dxs[r,d] = bf16(sum_n dz[r,n] * wi[e,d,n]): dz along 2F, wi
 *              along its last axis (wq_bwd of moe_mx_quantize_wi);
 *   wgrads     dwo[e,f,d] = bf16(sum_{r in e} h[r,f] * dys[r,d]) and
 *              dwi[e,d,n] = bf16(sum_{r in e} xs[r,d] * dz[r,n]): both
 *              operands quantized along the tokens of each group
 *              (moe_mx_quantize_tokens), in 32-row blocks from the group's
 *              first row (a group's last block may be short; it is padded
 *              with zeros); an expert without rows gets zeros.
 * The quantized tensors are the bf16 ones the block keeps (xs, h, z) and
 * the bf16 gradients (dys from moe_combine_bwd, dz).
 *
 * Layouts.  Weights quantized along their last axis keep their own layout,
 * codes [E, N, k] (wi: N = D, k = 2F; wo: N = F, k = D), with scales
 * [E, KB(k), NBp(N), 512] (the weight layout above without a transpose).
 * Row-quantized gradients use the activation layout above (codes [R, C],
 * tile-blocked scales).  Token-axis operands are stored transposed: with
 * TB = ceil(R/128) + E tiles and Rp = 128 * TB, codes [C, Rp] where the
 * rows of group e fill token columns 128 * tb[e] + i (i < size_e; tb as
 * for tile-blocked scales; the rest of each tile is zero codes, and a
 * 32-token step of padding only has the scale of a zero block, byte 0), and scales
 * [TB, NBp(C), 512]: tile g's scales for rows c of block c / 128 are the
 * block at ((g * NBp(C)) + c / 128) * 512, byte (c % 128 % 32) * 16 +
 * (c % 128 / 32) * 4 + j for tokens [32j, 32j+32) of the tile.
 */
/* The combine backward (moe_combine_bwd: dys bf16 [R, D] and dw) that also
 * writes dys quantized along D for the FC2 dgrad, dyq [R, D] with the
 * tile-blocked scales dysc, the bytes moe_mx_quantize_rows would make of
 * the same dys, without reading it back.  group_offsets: those of the
 * histogram that produced pos. */
moe_status moe_mx_combine_bwd(const moe_bf16* dout, const moe_bf16* ys, const float* w,
                              const int32_t* pos, const int32_t* group_offsets, moe_bf16* dys,
                              uint8_t* dyq, uint8_t* dysc, float* dw, moe_dims d,
                              cudaStream_t stream);
/* src bf16 [R, C] in expert-sorted order (C = D for dys, 2F for dz) -> q
 * [R, C] codes and tile-blocked scales sc (blocks along C). */
moe_status moe_mx_quantize_rows(const moe_bf16* src, int C, const int32_t* group_offsets,
                                uint8_t* q, uint8_t* sc, moe_dims d, cudaStream_t stream);
/* Token-axis quantization of src bf16 [R, C] in expert-sorted order, or,
 * when row_src is given, of the token-major x [T, C] read at token
 * row_src[r] / K for sorted row r (xs without its permuted copy).  C is D,
 * F or 2F.  qt [C, Rp] and sct as described above. */
moe_status moe_mx_quantize_tokens(const moe_bf16* src, const int32_t* row_src, int C,
                                  const int32_t* group_offsets, uint8_t* qt, uint8_t* sct,
                                  moe_dims d, cudaStream_t stream);
/* FC2 backward: dz from (dyq, dysc) and (woq, wosc) = wq_bwd of moe_mx_quantize_wo
 * and z; dwo bf16 [E, F, D] from ht/htsc (h along tokens) and dyt/dytsc
 * (dys along tokens).  dz and dwo may each be NULL (their inputs then too),
 * not both. */
moe_status moe_mx_grouped_gemm_fc2_bwd(const uint8_t* dyq, const uint8_t* dysc,
                                       const uint8_t* woq, const uint8_t* wosc, const moe_bf16* z,
                                       const uint8_t* ht, const uint8_t* htsc,
                                       const uint8_t* dyt, const uint8_t* dytsc,
                                       const int32_t* group_offsets, moe_bf16* dz, moe_bf16* dwo,
                                       int32_t* dev_status, moe_dims d, cudaStream_t stream);
/* FC1 backward: dxs bf16 [R, D] from (dzq, dzsc) and (wiq, wisc) of
 * moe_mx_quantize_wi (wq_bwd); dwi bf16 [E, D, 2F] from xt/xtsc (xs along
 * tokens) and dzt/dztsc (dz along tokens).  Either output may be NULL. */
moe_status moe_mx_grouped_gemm_fc1_bwd(const uint8_t* dzq, const uint8_t* dzsc,
                                       const uint8_t* wiq, const uint8_t* wisc,
                                       const uint8_t* xt, const uint8_t* xtsc,
                                       const uint8_t* dzt, const uint8_t* dztsc,
                                       const int32_t* group_offsets, moe_bf16* dxs, moe_bf16* dwi,
                                       int32_t* dev_status, moe_dims d, cudaStream_t stream);

/*
 * Fused forward for inference [Fused MoE Summary: gather, GMM1, activation
 * and GMM2 in one pass; Fused p/c Commits table row 1: the combine as the
 * unpermute plus the top-K weighted sum].  After moe_route_histogram, the
 * block's forward without the permuted copy xs and without ys:
 *   h = silu(a[:F]) * a[F:], a = x[row_src[r] / K] . wi[e]   (FC1 on rows
 *       gathered from the token-major x; the sorted order is row_src's)
 *   out[t] = bf16(sum_k w[t,k] * (h[pos[t,k]] . wo[e]))       (FC2 with the
 *       weighted combine in its epilogue, summed in fp32 in acc)
 *   x bf16 [T,D], w fp32 [T,K], row_src int32 [R] and group_offsets [E+1]
 *   from moe_route_histogram, wi, wo as for the unfused calls;
 *   h    bf16 [R,F]  scratch (FC1's output, FC2's input), caller-owned;
 *   acc  fp32 [T,D]  scratch, caller-owned (zeroed by the call);
 *   out  bf16 [T,D]  out.
 * Rows of row_src that are -1 (dropped slots) contribute nothing.  The fp32
 * sums of the combine are added in an unspecified order, so out is not
 * bitwise reproducible between runs; each element is within the block's
 * tolerance of the unfused moe_combine result (which rounds each ys to bf16
 * first).  No z is produced: this is the inference forward.
 */
moe_status moe_fused_forward(const moe_bf16* x, const float* w, const int32_t* row_src,
                             const int32_t* group_offsets, const moe_bf16* wi, const moe_bf16* wo,
                             moe_bf16* h, float* acc, moe_bf16* out, int32_t* dev_status,
                             void* ws, moe_dims d, cudaStream_t stream);

/*
 * Self-test of the kernels' bounded waits (no counterpart on the pages):
 * launches one block that waits on a barrier nothing ever arrives at, with a
 * limit of `limit_ns` nanoseconds (at most 10^9).  The wait gives up,
 * MOE_ERR_TIMEOUT is written to *dev_status and the kernel returns normally,
 * leaving the context usable.
 */
moe_status moe_selftest_bounded_wait(int32_t* dev_status, uint64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
