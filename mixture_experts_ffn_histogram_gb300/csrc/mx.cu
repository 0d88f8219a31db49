// MXFP8 forward of the MoE block on the fifth-generation tensor cores.
//
// What is computed (TransformerEngine "[DRAFT][JAX] Optimize MoE block",
// Changes item 1: MXFP8 quantization in the MoE block; Flowchart: "Grouped
// FC1 quantize and GEMM" -> "Activation and grouped FC2 GEMM"), with MXFP8
// read as the OCP MX v1.0 format: blocks of 32 elements along the
// contraction axis share an E8M0 scale 2^s, s = max(floor(log2 amax) - 8,
// -127); elements are E4M3 codes of v / 2^s, nearest-even, saturating.
//   grouped quantize   the expert weights (once, transposed so that the
//                      contraction axis is contiguous) and the tokens while
//                      they are gathered into expert-sorted order
//   FC1 + SwiGLU       h = silu(a[:F]) * a[F:], a = x . wi[e] on MX operands,
//                      h quantized to MX in the epilogue for FC2
//   FC2                ys = h . wo[e] on MX operands, bf16 output
//
// GEMM design: persistent warp-specialised kernel, one CTA per SM, 192
// threads, 128-row x 256-column tiles, k-blocks of 128 fp8 elements.
//   warp 0     producer: per k-block one TMA box of A (128 x 128 B), one of
//              B (256 x 128 B, 128-byte swizzle) and two bulk copies of the
//              tile's scale blocks (512 B for A, 1 KB for B) into a 4-deep
//              shared-memory ring.
//   warp 1     TMEM allocation and MMA issue by one thread: per k-block the
//              scale blocks are copied into TMEM (tcgen05.cp) and each
//              32-element k-step issues one block-scaled MMA (M = 128,
//              N = 256).  The thread's issue rate bounds the kernel: two
//              N = 128 MMAs per k-step took 25% longer, and per-k-step
//              descriptor arithmetic and warp votes cost 15% more, so the
//              descriptors are stage bases plus constant offsets and no other
//              lane takes part.
//   warps 2-5  epilogue: one row per thread (tcgen05.ld), SwiGLU and MX
//              quantization of h (FC1) or bf16 conversion (FC2), TMA stores
//              from per-warp staging.
// TMEM: two 256-column accumulators; the tile in one keeps its scale slots
// (16 columns per ring stage, 64 in all) in the first columns of the other,
// which the epilogue reads first and releases early (sffree), so the next
// tile waits only for that half of the previous tile's accumulator.  (Two
// whole accumulators would leave no columns for scales otherwise.)
// The scale-factor layout in TMEM (checked on GB300 by an in-bounds probe
// whose scale bytes encoded their own positions): for 128 rows and a
// 128-element k-block, the 512-byte block holds row m's scale for k-step j
// at byte (m % 32) * 16 + (m / 32) * 4 + j; tcgen05.cp.32x128b.warpx4 places
// it in four TMEM columns and the instruction descriptor's scale ids pick j.
// For N = 256 the B scales of rows 128-255 are the next block, four columns on.
#include <cuda.h>
#include <cuda_fp8.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "mx.h"
#include "mx_common.cuh"

namespace moe {

namespace {

constexpr int kMaxE = 1024;
constexpr int kThreads = 192;
constexpr int kMaxStages = 4;
constexpr int kAStage = 128 * 128;               // 16 KB
constexpr int kBStage = 256 * 128;               // 32 KB
constexpr int kSfaOff = kAStage + kBStage;       // 48 KB
constexpr int kSfbOff = kSfaOff + 1024;
constexpr int kStageBytes = kSfbOff + 1024;      // 50 KB (keeps every operand 1024-aligned)
constexpr uint32_t kTxBytes = kAStage + kBStage + 512 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfStride = 16;               // scale slot per stage: A 4 + B 8 columns (16-aligned)

// How many of the first n uses of a ring of S stages (taken in order) fell
// on stage i: one counter per ring instead of a per-stage array, which a
// run-time index would put in local memory.
__device__ __forceinline__ uint32_t mx_ring_uses(uint32_t n, uint32_t i, uint32_t S) {
  return n > i ? (n - i + S - 1) / S : 0u;
}

struct MxCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];   // accumulator buffer b holds a finished tile
  uint64_t tempty[2];  // the epilogue has read all of buffer b
  uint64_t sffree[2];  // the epilogue has read half 0 of buffer b (the scale slots)
  uint64_t zbar[4][2]; // FC2 dgrad: z chunk slot s of epilogue warp w has landed
  uint32_t tmem_base;
  int abort_flag;
  int off[kMaxE + 1];  // group offsets
  int tb[kMaxE + 1];   // first 128-row tile of each group (exclusive prefix)
};
// Per tile kind: ring stages and staging bytes per epilogue warp.  The FC2
// dgrad gives up a ring stage for two 8 KB slots per epilogue warp, each
// holding a 64-column chunk of z's gate and up halves (TMA loads) that the
// SwiGLU backward turns into dz in place (TMA stores).
template <int KIND>
struct MxCfg {
  static constexpr int kStages = KIND == 2 ? 3 : 4;
  static constexpr int kEpiBytes = KIND == 2 ? 16384 : 4096;
  static constexpr size_t kSmemBytes =
      1024 + static_cast<size_t>(kStages) * kStageBytes + 4 * kEpiBytes + sizeof(MxCtl);
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// ------------------------------------------------- transpose-quantize
// MX quantization along the ROWS of a bf16 matrix tile of 128 rows x 128
// columns, stored transposed: each column's 128 values form four 32-element
// blocks; a thread takes two adjacent columns of one block (one 32-bit
// shared-memory read per row gives both, and their largest magnitudes come
// from packed integer maxima of the bf16 bits).  The input tile is staged
// in shared memory as bf16 (32 KB), copied with 16-byte cp.async row
// segments (a warp reads two 256-byte row pieces); the codes are gathered
// into a 128-byte-swizzled output tile (a row per column) that two TMA
// stores write out, 64 output rows each (writing each column's 32 codes
// from its own thread touched 32 lines per warp store and ran at half the
// HBM rate).
// Two uses:
//   tokens   rows = 128 expert-sorted rows of tile g of group e (rows past
//            the group's end as zeros), read in place or gathered from x at
//            token row_src[r] / K: codes qt[c][128 g .. 128 g + 127], scales
//            [TB][NBp(C)][512] block (g, c / 128);
//   weights  rows = k-block kb of expert e of w [E][Kd][N] (rows past Kd as
//            zeros): codes q[e][p(n)][Kd] with 128 (or, at a ragged last
//            k-block, 64) bytes per column, scales [E][KB][NBp][512]; FC1's
//            output rows are interleaved in 64-row chunks, gate chunk then up
//            chunk: column n of wi (gate f = n < F, up f = n - F) lands on
//            row p = 128 (f / 64) + 64 (n >= F) + f % 64, so that each
//            128-row half of a 256-row tile holds 64 gate and the matching
//            64 up columns.  Optionally the same tile also gives the weight
//            quantized along its LAST axis N (the dgrads' contraction axis),
//            codes in w's own layout and scales [E][KB(N)][NBp(Kd)][512].
constexpr int kTqRows = 128;
constexpr int kTqCols = 128;
constexpr int kTqThreads = 256;
constexpr int kTqBuf = kTqRows * kTqCols * 2;  // bytes of one staged input tile (32 KB)
constexpr int kTqOut = kTqCols * 128;          // the codes of one item: 128 columns x 128 B
// input double buffer, the output tile (two 64-row halves, 128-byte swizzled
// for the TMA store), one 512-byte scale block, and slack for 1024-alignment
constexpr int kTqSmem = 2 * kTqBuf + kTqOut + 512 + 1024;
constexpr int kTqCtasPerSm = 2;

struct TqArgs {
  const uint16_t* src;     // tokens: [R or T][C]; weights: w [E][Kd][N]
  const int32_t* row_src;  // tokens: gather through row_src[r] / K, or nullptr
  const int32_t* offs;     // tokens: group offsets
  uint8_t* q;              // transposed codes (see above), or nullptr (weights)
  uint8_t* sc;
  uint8_t* q2;             // weights: last-axis codes [E][Kd][N], or nullptr
  uint8_t* sc2;
  long Rp;                 // tokens: token columns of qt
  int C;                   // columns (tokens: C; weights: N)
  int K;                   // tokens: slots per token (row_src / K)
  int E;
  int Kd;                  // weights: rows per expert
  int KB;                  // weights: k-blocks of Kd
  int NBp;                 // 128-row scale blocks of the transposed output, even
  int KB2;                 // weights: k-blocks of N (last-axis scales)
  int NBp2;                // weights: 128-row blocks of Kd (last-axis scales)
  int interleave;          // weights: FC1 row interleave
};

// One work item: 128 source rows from row0 (rows of them valid) x 128
// columns from c0; tokens: tile g of group e; weights: k-block kb of expert e.
struct TqItem {
  long row0;
  int rows, c0, e, g, kb;
};

// Persistent: each CTA takes work items it = blockIdx.x, + gridDim.x, ...
// and copies the next item's tile into the other buffer (cp.async, rows past
// the valid ones zero-filled) while it quantizes the current one.
template <bool TOKENS>
__global__ void __launch_bounds__(kTqThreads, kTqCtasPerSm)
    mx_transpose_quantize_kernel(const __grid_constant__ CUtensorMap map_q, const TqArgs a) {
  extern __shared__ __align__(128) uint8_t tq_raw[];
  uint8_t* tq_smem = tq_raw + ((1024u - (smem_u32(tq_raw) & 1023u)) & 1023u);
  uint8_t* stage = tq_smem + 2 * kTqBuf;  // codes: [2 halves][64 rows][128 B], swizzled
  uint8_t* s_sc = stage + kTqOut;         // tokens: the item's scale block
  __shared__ int s_off[TOKENS ? kMaxE + 1 : 1];
  __shared__ int s_tb[TOKENS ? kMaxE + 1 : 1];
  const int tid = threadIdx.x;
  const int nchunks = (a.C + kTqCols - 1) / kTqCols;
  long n_items;
  if constexpr (TOKENS) {
    load_tile_bases(a.offs, a.E, s_off, s_tb, 0);
    n_items = static_cast<long>(s_tb[a.E]) * nchunks;
  } else {
    n_items = static_cast<long>(nchunks) * a.KB * a.E;
  }
  auto decode = [&](long it) {
    TqItem I;
    const int chunk = static_cast<int>(it % nchunks);
    const long rest = it / nchunks;
    I.c0 = chunk * kTqCols;
    if constexpr (TOKENS) {
      I.g = static_cast<int>(rest);
      int lo = 0, hi = a.E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_tb[mid] <= I.g) lo = mid;
        else hi = mid - 1;
      }
      I.e = lo;
      I.kb = 0;
      I.row0 = s_off[lo] + 128L * (I.g - s_tb[lo]);
      I.rows = min(128, static_cast<int>(s_off[lo + 1] - I.row0));
    } else {
      I.kb = static_cast<int>(rest % a.KB);
      I.e = static_cast<int>(rest / a.KB);
      I.g = 0;
      I.row0 = static_cast<long>(I.e) * a.Kd + 128L * I.kb;
      I.rows = min(128, a.Kd - 128 * I.kb);
    }
    return I;
  };
  // 128 rows x 16 16-byte segments: 8 per thread, a warp per two 256-byte
  // rows.  The source rows of an item (gathered: loaded from row_src) are
  // found one item before its copies are issued, so that no copy waits for
  // an index load.
  auto rows_of = [&](const TqItem& I, long (&sr)[8]) {
    const int seg = tid & 15;
    const bool col_ok = I.c0 + 8 * seg < a.C;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 16 * i + (tid >> 4);
      sr[i] = (r < I.rows && col_ok) ? I.row0 + r : -1;
      if (TOKENS && a.row_src != nullptr && sr[i] >= 0) sr[i] = __ldg(a.row_src + sr[i]);
    }
  };
  auto issue = [&](const long (&sr)[8], const TqItem& I, uint8_t* buf) {
    const int seg = tid & 15;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 16 * i + (tid >> 4);
      long row = sr[i];
      if (TOKENS && a.row_src != nullptr && row >= 0) row /= a.K;
      const uint16_t* src = row >= 0 ? a.src + row * a.C + I.c0 + 8 * seg : a.src;
      cp_async16_zfill(buf + r * (kTqCols * 2) + 16 * seg, src, row >= 0 ? 16 : 0);
    }
    cp_async_commit();
  };

  long it = blockIdx.x;
  if (it >= n_items) return;  // block-uniform
  if (tid == 0 && a.q != nullptr) tma_prefetch_map(&map_q);
  TqItem cur = decode(it);
  long sr_cur[8], sr_nxt[8];
  rows_of(cur, sr_cur);
  issue(sr_cur, cur, tq_smem);
  TqItem nxt = cur;
  if (it + gridDim.x < n_items) {
    nxt = decode(it + gridDim.x);
    rows_of(nxt, sr_nxt);
  }
  for (int k = 0; it < n_items; it += gridDim.x, ++k) {
    const long nx = it + gridDim.x;
    TqItem after = nxt;  // the item after the next one, and its rows
    long sr_after[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sr_after[i] = -1;
    if (nx < n_items) {
      issue(sr_nxt, nxt, tq_smem + ((k + 1) & 1) * kTqBuf);
      if (nx + gridDim.x < n_items) {
        after = decode(nx + gridDim.x);
        rows_of(after, sr_after);
      }
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    if (tid == 0) bulk_wait_read<0>();  // the previous item's stores have read the stage
    __syncthreads();
    const uint8_t* tile = tq_smem + (k & 1) * kTqBuf;
    // ---- two adjacent columns and one 32-row block per thread; the codes go
    // to the swizzled output tile (row = column), written by two TMA stores
    if (a.q != nullptr) {
      const int cp = tid & 63, b = tid >> 6;
      const int cl = 2 * cp;
      const int c = cur.c0 + cl;
      uint32_t ca[8], cb[8], sab = 0;
      const bool ok = c < a.C && (TOKENS || 32 * b < cur.rows);
      // (tokens: rows past the group's end are quantized too, giving zero
      // codes and the zero block's scale; weights: rows past Kd are clipped
      // by the store)
      if (ok) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          w[i] = *reinterpret_cast<const uint32_t*>(tile + (32 * b + i) * (kTqCols * 2) + 4 * cp);
        sab = mx_quant_col2(w, ca, cb);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) ca[i] = cb[i] = 0u;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = cl + h;  // output tile row (0..127)
        const uint32_t* cw = h ? cb : ca;
        uint8_t* rbase = stage + (row >> 6) * (kTqOut / 2) + (row & 63) * 128;
        *reinterpret_cast<uint4*>(rbase + (((2 * b) ^ (row & 7)) << 4)) =
            make_uint4(cw[0], cw[1], cw[2], cw[3]);
        *reinterpret_cast<uint4*>(rbase + (((2 * b + 1) ^ (row & 7)) << 4)) =
            make_uint4(cw[4], cw[5], cw[6], cw[7]);
        const uint8_t sbyte = static_cast<uint8_t>(sab >> (8 * h));
        if constexpr (TOKENS) {
          s_sc[sf_byte(row, b)] = sbyte;
        } else if (ok) {
          const int cc = c + h;
          int p = cc;
          if (a.interleave) {
            const int F = a.C / 2;
            const int f = cc < F ? cc : cc - F;
            p = 128 * (f >> 6) + (cc < F ? 0 : 64) + (f & 63);
          }
          const size_t sblk = (static_cast<size_t>(cur.e) * a.KB + cur.kb) * a.NBp + (p >> 7);
          a.sc[sblk * 512 + sf_byte(p & 127, b)] = sbyte;
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        for (int hh = 0; hh < 2; ++hh) {
          const int cf = cur.c0 + 64 * hh;  // first column of the half
          if (cf >= a.C) break;
          if constexpr (TOKENS) {
            tma_store_2d(&map_q, stage + hh * (kTqOut / 2), 128 * cur.g, cf);
          } else {
            int p0 = cf;
            if (a.interleave) {
              const int F = a.C / 2;
              const bool up = cf >= F;
              p0 = 128 * ((cf - (up ? F : 0)) >> 6) + (up ? 64 : 0);
            }
            tma_store_2d(&map_q, stage + hh * (kTqOut / 2), 128 * cur.kb, cur.e * a.C + p0);
          }
        }
        bulk_commit();
      }
      if constexpr (TOKENS) {
        if (tid < 32) {
          const size_t sblk = static_cast<size_t>(cur.g) * a.NBp + (cur.c0 >> 7);
          reinterpret_cast<uint4*>(a.sc + sblk * 512)[tid] =
              reinterpret_cast<const uint4*>(s_sc)[tid];
        }
      }
    }
    if constexpr (!TOKENS) {
      // ---- the same tile along its last axis: 4 blocks of 32 columns per row
      if (a.q2 != nullptr) {
        for (int id = tid; id < kTqRows * 4; id += kTqThreads) {
          const int r = id >> 2, nb = id & 3;
          const int n0 = cur.c0 + 32 * nb;
          if (r >= cur.rows || n0 >= a.C) continue;
          uint32_t w[16];
          const uint4* src4 = reinterpret_cast<const uint4*>(tile + r * (kTqCols * 2) + 64 * nb);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 u = src4[i];
            w[4 * i] = u.x;
            w[4 * i + 1] = u.y;
            w[4 * i + 2] = u.z;
            w[4 * i + 3] = u.w;
          }
          uint32_t codes[8];
          const uint32_t sbyte = mx_quant_row32(w, codes);
          const long kr = 128L * cur.kb + r;  // row of the expert
          uint4* d4 =
              reinterpret_cast<uint4*>(a.q2 + (static_cast<size_t>(cur.e) * a.Kd + kr) * a.C + n0);
          d4[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
          d4[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
          const size_t blk =
              (static_cast<size_t>(cur.e) * a.KB2 + (n0 >> 7)) * a.NBp2 + (kr >> 7);
          a.sc2[blk * 512 + sf_byte(static_cast<int>(kr & 127), (n0 & 127) >> 5)] =
              static_cast<uint8_t>(sbyte);
        }
      }
    }
    __syncthreads();  // the input buffer is refilled two items on
    cur = nxt;
    nxt = after;
#pragma unroll
    for (int i = 0; i < 8; ++i) sr_nxt[i] = sr_after[i];
  }
  if (tid == 0) bulk_wait_all();
}

// ------------------------------------------------ permute + quantize
// xq[pos[t,k]] = codes of x[t] (each token row quantized once, written K
// times); the scales go to the tile-blocked layout of the destination row:
// block (tb[e] + i/128) * KB + k-block, row i % 128, where i is the row's
// index inside its group e.  One warp per token; lane l quantizes 32-element
// blocks l, l+32, ...; the loads of kPqIt such rounds are issued before any
// is quantized, and each round's codes are redistributed by shuffles so that
// every store of the K copies writes 512 contiguous bytes (storing each
// block's 32 bytes from its own lane took 25% longer).
constexpr int kPqWarps = 8;
constexpr int kPqIt = 2;
__global__ void __launch_bounds__(256) mx_permute_quantize_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ pos,
    const int32_t* __restrict__ offs, uint8_t* __restrict__ xq, uint8_t* __restrict__ xsc, int T,
    int D, int K, int E, int KB) {
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_tb[kMaxE + 1];
  __shared__ int s_row[kPqWarps][32];
  __shared__ int s_blk[kPqWarps][32];  // scale block base (bytes) of the slot's row
  __shared__ int s_m[kPqWarps][32];
  load_tile_bases(offs, E, s_off, s_tb, 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = D / 32;
  const int R = s_off[E];
  for (int t = blockIdx.x * kPqWarps + warp; t < T; t += gridDim.x * kPqWarps) {
    if (lane < K) {
      // pos == nullptr: the rows are already in sorted order (K == 1)
      int r = pos != nullptr ? __ldg(pos + static_cast<size_t>(t) * K + lane) : t;
      if (r >= R) r = -1;
      int blk = 0, m = 0;
      if (r >= 0) {
        const int e = group_of_row(s_off, E, r);
        const int i = r - s_off[e];
        blk = (s_tb[e] + (i >> 7)) * KB;
        m = i & 127;
      }
      s_row[warp][lane] = r;
      s_blk[warp][lane] = blk;
      s_m[warp][lane] = m;
    }
    __syncwarp();
    const uint16_t* xr = x + static_cast<size_t>(t) * D;
    // up to kPqIt 32-block rounds of the row are loaded before any is
    // quantized, so their memory latencies overlap
    for (int b0 = 0; b0 < nb; b0 += 32 * kPqIt) {
      uint4 u[kPqIt][4];
#pragma unroll
      for (int j = 0; j < kPqIt; ++j) {
        const int b = b0 + 32 * j + lane;
        if (b < nb) {
          const uint4* src = reinterpret_cast<const uint4*>(xr + 32 * b);
#pragma unroll
          for (int i = 0; i < 4; ++i) u[j][i] = src[i];
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) u[j][i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int j = 0; j < kPqIt; ++j) {
        const int b = b0 + 32 * j + lane;
        if (b0 + 32 * j >= nb) break;  // warp-uniform: the round is empty
        float v[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t wv[4] = {u[j][i].x, u[j][i].y, u[j][i].z, u[j][i].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            v[8 * i + 2 * q] = bf16lo(wv[q]);
            v[8 * i + 2 * q + 1] = bf16hi(wv[q]);
          }
        }
        uint32_t codes[8];
        const uint8_t sbyte = static_cast<uint8_t>(mx_quant32(v, codes));
        // redistribute the round's codes (lane l holds block b0' + l) so
        // that each warp store writes 512 contiguous bytes: in store h,
        // lane l writes half (l & 1) of block b0' + 16h + (l >> 1)
        uint4 out[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int src = 16 * h + (lane >> 1);
          uint32_t lo[4], hi[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            lo[i] = __shfl_sync(0xffffffffu, codes[i], src);
            hi[i] = __shfl_sync(0xffffffffu, codes[4 + i], src);
          }
          out[h] = (lane & 1) ? make_uint4(hi[0], hi[1], hi[2], hi[3])
                              : make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        const int rb = b - lane;  // first block of the round
        for (int k = 0; k < K; ++k) {
          const int r = s_row[warp][k];
          if (r < 0) continue;
          uint8_t* row = xq + static_cast<size_t>(r) * D + 32 * rb;
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (rb + 16 * h + (lane >> 1) < nb)
              *reinterpret_cast<uint4*>(row + 512 * h + 16 * lane) = out[h];
          if (b < nb) {
            const size_t blk = static_cast<size_t>(s_blk[warp][k]) + (b >> 2);
            xsc[blk * 512 + sf_byte(s_m[warp][k], b & 3)] = sbyte;
          }
        }
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- GEMM
constexpr int kKFc1 = static_cast<int>(MxKind::kFc1);
constexpr int kKRows = static_cast<int>(MxKind::kRows);
constexpr int kKSwigluBwd = static_cast<int>(MxKind::kRowsSwigluBwd);
constexpr int kKWgrad = static_cast<int>(MxKind::kWgrad);

struct MxParams {
  const uint8_t* sfa;   // A scales, tile-blocked [tiles][KB][512]
  const uint8_t* sfb;   // B scales [E][KB][NBp][512]
  const int32_t* offs;
  uint8_t* hq;          // FC1: h codes [R][F] or nullptr
  uint8_t* hsc;         // FC1: h scales, tile-blocked [tiles][KBF][512]
  __nv_bfloat16* out;   // FC1: h bf16 [R][F] or nullptr; rows: [R][Nout]; SwiGLU
                        // backward: dz [R][2 Nout]; wgrad: [E][Ma][Nout]
  const __nv_bfloat16* zin;  // SwiGLU backward: z [R][2 Nout]
  __nv_bfloat16* zout;  // FC1: z [R][2F] or nullptr
  int32_t* status;
  uint64_t limit_ns;
  int E;
  int Kd;       // contraction length (rows kinds; a bound on it for the wgrad)
  int KB;       // k-blocks of Kd
  int Nout;     // output columns: FC1 F (h columns); others the B rows per expert
  int NBp;      // 128-row blocks of B per (expert or token tile, k-block), even
  int n_tiles;  // 256-row B tiles per expert
  int KBF;      // FC1: k-blocks of F (h scale blocks per tile row)
  int Ma;       // wgrad: output rows per expert (A rows)
  int m_tiles;  // wgrad: 128-row A tiles
  int NBpA;     // wgrad: 128-row blocks of A per token tile
};

// One output tile: expert e, B tile nt; rows kinds: sorted-row tile g whose
// rows row0 .. row0 + rows - 1 are A's and the output's; wgrad: A tile mt,
// output rows row0 = e * Ma + 128 mt ..; the k-blocks kb0 .. kb0 + nkb - 1.
struct MxTile {
  int e, g, nt, mt, row0, rows, kb0, nkb;
};

template <int KIND>
__device__ __forceinline__ MxTile mx_decode(int t, const MxParams& p, const MxCtl& s) {
  MxTile T;
  if constexpr (KIND == kKWgrad) {
    T.nt = t % p.n_tiles;
    const int em = t / p.n_tiles;
    T.mt = em % p.m_tiles;
    T.e = em / p.m_tiles;
    T.g = 0;
    T.row0 = T.e * p.Ma + 128 * T.mt;
    T.rows = min(128, p.Ma - 128 * T.mt);
    T.kb0 = s.tb[T.e];
    T.nkb = s.tb[T.e + 1] - T.kb0;
    return T;
  }
  T.mt = 0;
  T.kb0 = 0;
  T.nkb = p.KB;
  T.g = t / p.n_tiles;
  T.nt = t - T.g * p.n_tiles;
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.tb[mid] <= T.g) lo = mid;
    else hi = mid - 1;
  }
  T.e = lo;
  T.row0 = s.off[lo] + (T.g - s.tb[lo]) * 128;
  T.rows = min(128, s.off[lo + 1] - T.row0);
  return T;
}

// Whether half h (128 B rows) of tile nt holds any output column.
template <int KIND>
__device__ __forceinline__ bool half_valid(int nt, int h, const MxParams& p) {
  return KIND == kKFc1 ? 64 * (2 * nt + h) < p.Nout : 256 * nt + 128 * h < p.Nout;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Descriptor of a 512-byte scale block in shared memory (32 rows of 16 B,
// no swizzle) for tcgen05.cp.
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>(128 >> 4) << 32) | (1ull << 46);
}
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// Block-scaled MMA: e4m3 A (M = 128) and B (N = 128), both K-major, K = 32,
// E8M0 scales at sfa/sfb in TMEM.
__device__ __forceinline__ void umma_mxf8(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc,
                                          uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// Instruction descriptor, kind::mxf8f6f4 with block scaling: B scale id in
// bits 4-5, A and B formats e4m3 (0) in bits 7-9 and 10-12, K-major A and
// B, N >> 3 in bits 17-22, E8M0 scales (bit 23), M >> 4 in bits 24-28, A
// scale id in bits 29-30.
__host__ __device__ constexpr uint32_t mx_idesc(int M, int N, int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4) | ((static_cast<uint32_t>(N) >> 3) << 17) |
         (1u << 23) | ((static_cast<uint32_t>(M) >> 4) << 24) |
         (static_cast<uint32_t>(sf_id) << 29);
}

__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// 16 packed bf16 pairs = 32 columns (half `hh` of a 64-column row) of row
// `lane` in a 128-byte-swizzled staging buffer.
__device__ __forceinline__ void put_half_sw(uint8_t* buf, int lane, int hh, const uint32_t (&w)[16]) {
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int unit = hh * 4 + j;
    *reinterpret_cast<uint4*>(row + ((unit ^ (lane & 7)) << 4)) =
        make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

// map_z, map_h: FC1 in training, z [R][2F] and the bf16 h [R][F] (64 x 32
// boxes, 128-byte swizzle); other kinds get copies of map_o, unused.
template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_o,
                   const __grid_constant__ CUtensorMap map_z,
                   const __grid_constant__ CUtensorMap map_h, const MxParams p) {
  using C = MxCfg<KIND>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* epi = ring + C::kStages * kStageBytes;
  MxCtl& s = *reinterpret_cast<MxCtl*>(epi + 4 * C::kEpiBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_a);
    tma_prefetch_map(&map_b);
    tma_prefetch_map(&map_o);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 4);
      mbar_init(&s.sffree[i], 4);
    }
    for (int w = 0; w < 4; ++w)
      for (int i = 0; i < 2; ++i) mbar_init(&s.zbar[w][i], 1);
    s.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc<1>(&s.tmem_base, kTmemCols);
    tmem_relinquish<1>();
  }
  load_tile_bases(p.offs, p.E, s.off, s.tb, 2);  // ends with __syncthreads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  const WaitCtl wc{&s.abort_flag, p.status, p.limit_ns};
  const int ntiles =
      KIND == kKWgrad ? p.E * p.m_tiles * p.n_tiles : s.tb[p.E] * p.n_tiles;

  if (warp == 0) {
    // -------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, nfill = 0;  // stages filled so far
      bool aborted = false;
      for (int t = blockIdx.x; t < ntiles && !aborted; t += gridDim.x) {
        const MxTile T = mx_decode<KIND>(t, p, s);
        const uint8_t* sfa;
        const uint8_t* sfb;
        size_t sfa_step;
        if constexpr (KIND == kKWgrad) {
          sfa = p.sfa + (static_cast<size_t>(T.kb0) * p.NBpA + T.mt) * 512;
          sfb = p.sfb + (static_cast<size_t>(T.kb0) * p.NBp + 2 * T.nt) * 512;
          sfa_step = static_cast<size_t>(p.NBpA) * 512;
        } else {
          sfa = p.sfa + static_cast<size_t>(T.g) * p.KB * 512;
          sfb = p.sfb + (static_cast<size_t>(T.e) * p.KB * p.NBp + 2 * T.nt) * 512;
          sfa_step = 512;
        }
        for (int kb = 0; kb < T.nkb; ++kb) {
          if (!mbar_wait(&s.empty[stage], phase ^ 1u, wc)) { aborted = true; break; }
          uint8_t* st = ring + stage * kStageBytes;
          mbar_arrive_expect_tx(&s.full[stage], kTxBytes);
          const int kx = (T.kb0 + kb) * 128;
          if constexpr (KIND == kKWgrad) {
            tma_load_2d(st, &map_a, &s.full[stage], kx, 128 * T.mt);
            tma_load_3d(st + kAStage, &map_b, &s.full[stage], kx, 256 * T.nt, 0);
          } else {
            tma_load_2d(st, &map_a, &s.full[stage], kx, T.row0);
            tma_load_3d(st + kAStage, &map_b, &s.full[stage], kx, 256 * T.nt, T.e);
          }
          bulk_load(st + kSfaOff, sfa + kb * sfa_step, 512, &s.full[stage]);
          bulk_load(st + kSfbOff, sfb + static_cast<size_t>(kb) * p.NBp * 512, 1024,
                    &s.full[stage]);
          ++nfill;
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (aborted) {  // copies in flight land before the CTA exits
        for (uint32_t i = 0; i < C::kStages; ++i) {
          const uint32_t f = mx_ring_uses(nfill, i, C::kStages);
          if (f > 0) (void)mbar_wait_drain(&s.full[i], (f - 1u) & 1u, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA
    // one thread: waits, scale copies, MMAs and commits
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, it = 0;
      uint32_t ncommit = 0;  // stages whose MMAs were committed so far
      bool aborted = false;
      // descriptors of stage 0's A and scale blocks; stage i adds i * kStageBytes >> 4,
      // a k-step 2 (32 B >> 4)
      const uint64_t da0 = smem_desc_sw128(smem_u32(ring), 16, 1024);
      const uint64_t ds0 = sf_desc(smem_u32(ring) + kSfaOff);
      for (int t = blockIdx.x; t < ntiles && !aborted; t += gridDim.x, ++it) {
        const MxTile T = mx_decode<KIND>(t, p, s);
        const bool h1 = half_valid<KIND>(T.nt, 1, p);
        // tile it accumulates in buffer it % 2 (256 columns) while its scale
        // slots sit in the first kStages * kSfStride columns of the other buffer, which
        // the epilogue empties first
        const uint32_t buf = it & 1u, use = it >> 1;
        if (!mbar_wait(&s.tempty[buf], (use & 1u) ^ 1u, wc) ||
            (it > 0 && !mbar_wait(&s.sffree[buf ^ 1u], ((it - 1) >> 1) & 1u, wc))) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + 256 * buf;
        const uint32_t sf_base = tmem_base + 256 * (buf ^ 1u);
        const uint32_t idn = h1 ? 256u : 128u;
        for (int kb = 0; kb < T.nkb; ++kb) {
          if (!mbar_wait(&s.full[stage], phase, wc)) { aborted = true; break; }
          tc_fence_after();
          const uint32_t sf = sf_base + kSfStride * stage;
          const uint64_t a0 = da0 + stage * (kStageBytes >> 4);
          const uint64_t b0 = a0 + (kAStage >> 4);
          const uint64_t s0 = ds0 + stage * (kStageBytes >> 4);
          tmem_cp_sf(sf, s0);
          tmem_cp_sf(sf + 4, s0 + (1024 >> 4));
          if (h1) tmem_cp_sf(sf + 8, s0 + (1536 >> 4));
          if (kb * 128 + 128 <= p.Kd) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
              umma_mxf8(d0, a0 + 2 * kk, b0 + 2 * kk, mx_idesc(128, idn, kk), sf, sf + 4, acc);
            }
          } else {
            const int nk = (p.Kd - kb * 128) / 32;
            for (int kk = 0; kk < nk; ++kk) {
              const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
              umma_mxf8(d0, a0 + 2 * kk, b0 + 2 * kk, mx_idesc(128, idn, kk), sf, sf + 4, acc);
            }
          }
          umma_commit<1>(&s.empty[stage]);
          ++ncommit;
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (aborted) break;
        umma_commit<1>(&s.tfull[buf]);
      }
      if (aborted && ncommit > 0) {  // issued MMAs finish before TMEM is freed
        const uint32_t last = (ncommit - 1u) % C::kStages;
        (void)mbar_wait_drain(&s.empty[last], (mx_ring_uses(ncommit, last, C::kStages) - 1u) & 1u,
                              100000000ull);
      }
    }
  } else {
    // -------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter: rows 32q..32q+31 of the tile
    const int ew = warp - 2;  // epilogue warp index
    uint8_t* buf = epi + ew * C::kEpiBytes;
    uint32_t it = 0;
    bool aborted = false;
    // FC2 dgrad, full warps: z chunk c (64 columns f = 256 nt + 64 c, gate
    // and up) lands in slot c & 1 by TMA; zpar / zout track each slot's
    // mbarrier phase and whether a load is outstanding
    uint32_t zpar[2] = {0u, 0u};
    bool zout[2] = {false, false};
    auto zload = [&](int slot, int f, int yrow) {
      uint8_t* dst = buf + slot * 8192;
      mbar_arrive_expect_tx(&s.zbar[ew][slot], 8192);
      tma_load_2d(dst, &map_z, &s.zbar[ew][slot], f, yrow);
      tma_load_2d(dst + 4096, &map_z, &s.zbar[ew][slot], p.Nout + f, yrow);
    };
    for (int t = blockIdx.x; t < ntiles && !aborted; t += gridDim.x, ++it) {
      const MxTile T = mx_decode<KIND>(t, p, s);
      const int vw = min(32, max(0, T.rows - 32 * q));  // valid rows of this warp
      const int y = T.row0 + 32 * q;
      const bool row_ok = lane < vw;
      const long r = static_cast<long>(y) + lane;
      const uint32_t bsel = it & 1u;
      const bool tma_z = KIND == kKSwigluBwd && vw == 32;
      if (tma_z) {  // z's first two chunks, requested before the accumulator is ready
        if (lane == 0) {
          bulk_wait_read<0>();  // the previous tile's dz stores have read the slots
          for (int c = 0; c < 2; ++c)
            if (256 * T.nt + 64 * c < p.Nout) zload(c, 256 * T.nt + 64 * c, y);
        }
        for (int c = 0; c < 2; ++c) zout[c] = 256 * T.nt + 64 * c < p.Nout;
        __syncwarp();
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&s.tfull[bsel], (it >> 1) & 1u, wc))) {
        aborted = true;
        break;
      }
      tc_fence_after();
      for (int hh = 0; hh < 2; ++hh) {
        const bool live = half_valid<KIND>(T.nt, hh, p) && vw > 0;
        // a wgrad tile of an empty group has no accumulator: its rows are zeros
        const bool empty = KIND == kKWgrad && T.nkb == 0;
        uint32_t v[128];
        if (live && !empty) {
          const uint32_t ta = tmem_base + 256 * bsel + 128 * hh + (static_cast<uint32_t>(32 * q) << 16);
          tmem_ld_32x32b_x32(ta, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld_32x32b_x32(ta + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_ld_32x32b_x32(ta + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[64]));
          tmem_ld_32x32b_x32(ta + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[96]));
          tmem_ld_wait();
        }
        // half 0 holds the next tile's scale slots (its first kStages * kSfStride
        // columns); half 1 ends this warp's reads of the buffer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(hh == 0 ? &s.sffree[bsel] : &s.tempty[bsel]);
        if (!live) continue;
        if constexpr (KIND == kKWgrad) {
          if (empty) {
            if (row_ok) {
              const int d0 = 256 * T.nt + 128 * hh;
              for (int col = d0; col < min(d0 + 128, p.Nout); col += 8)
                *reinterpret_cast<uint4*>(p.out + r * p.Nout + col) = make_uint4(0u, 0u, 0u, 0u);
            }
            continue;
          }
        }
        if constexpr (KIND == kKFc1) {
          // gate = columns 0..63, up = 64..127 of the region: h for f0..f0+63
          const int f0 = 64 * (2 * T.nt + hh);
          // a full warp stages z's gate and up chunks and h's bf16 chunk
          // through its swizzled buffer, one TMA store each (per-thread
          // stores of the same bytes cost the MMA: 1253 vs 794 us without
          // these outputs)
          if (vw == 32 && (p.zout != nullptr || (p.out != nullptr && p.hq != nullptr))) {
            for (int part = 0; part < 3; ++part) {
              if (part < 2 && p.zout == nullptr) continue;
              if (part == 2 && !(p.out != nullptr && p.hq != nullptr)) continue;
              uint32_t w0[16], w1[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float a0, a1, b0, b1;
                if (part < 2) {
                  const uint32_t* src = v + 64 * part;
                  a0 = __uint_as_float(src[2 * i]);
                  a1 = __uint_as_float(src[2 * i + 1]);
                  b0 = __uint_as_float(src[32 + 2 * i]);
                  b1 = __uint_as_float(src[32 + 2 * i + 1]);
                } else {
                  a0 = silu(__uint_as_float(v[2 * i])) * __uint_as_float(v[64 + 2 * i]);
                  a1 = silu(__uint_as_float(v[2 * i + 1])) * __uint_as_float(v[64 + 2 * i + 1]);
                  b0 = silu(__uint_as_float(v[32 + 2 * i])) * __uint_as_float(v[96 + 2 * i]);
                  b1 = silu(__uint_as_float(v[33 + 2 * i])) * __uint_as_float(v[97 + 2 * i]);
                }
                w0[i] = pack_bf16x2(a0, a1);
                w1[i] = pack_bf16x2(b0, b1);
              }
              if (lane == 0) bulk_wait_read<0>();
              __syncwarp();
              put_half_sw(buf, lane, 0, w0);
              put_half_sw(buf, lane, 1, w1);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (part == 0) tma_store_2d(&map_z, buf, f0, y);
                else if (part == 1) tma_store_2d(&map_z, buf, p.Nout + f0, y);
                else tma_store_2d(&map_h, buf, f0, y);
                bulk_commit();
              }
            }
          } else if (p.zout != nullptr && row_ok) {  // z = [gate | up] for the backward
            uint4* zg = reinterpret_cast<uint4*>(p.zout + r * 2 * p.Nout + f0);
            uint4* zu = reinterpret_cast<uint4*>(p.zout + r * 2 * p.Nout + p.Nout + f0);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t* a = v + 8 * i;
              zg[i] = make_uint4(pack_bf16x2(__uint_as_float(a[0]), __uint_as_float(a[1])),
                                 pack_bf16x2(__uint_as_float(a[2]), __uint_as_float(a[3])),
                                 pack_bf16x2(__uint_as_float(a[4]), __uint_as_float(a[5])),
                                 pack_bf16x2(__uint_as_float(a[6]), __uint_as_float(a[7])));
              const uint32_t* b = v + 64 + 8 * i;
              zu[i] = make_uint4(pack_bf16x2(__uint_as_float(b[0]), __uint_as_float(b[1])),
                                 pack_bf16x2(__uint_as_float(b[2]), __uint_as_float(b[3])),
                                 pack_bf16x2(__uint_as_float(b[4]), __uint_as_float(b[5])),
                                 pack_bf16x2(__uint_as_float(b[6]), __uint_as_float(b[7])));
            }
          }
          float hv[64];
#pragma unroll
          for (int j = 0; j < 64; ++j)
            hv[j] = silu(__uint_as_float(v[j])) * __uint_as_float(v[64 + j]);
          if (p.out != nullptr && row_ok && !(vw == 32 && p.hq != nullptr)) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + r * p.Nout + f0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_uint4(pack_bf16x2(hv[8 * i], hv[8 * i + 1]),
                                  pack_bf16x2(hv[8 * i + 2], hv[8 * i + 3]),
                                  pack_bf16x2(hv[8 * i + 4], hv[8 * i + 5]),
                                  pack_bf16x2(hv[8 * i + 6], hv[8 * i + 7]));
          }
          if (p.hq != nullptr) {
            uint32_t c[2][8];
            uint32_t sb[2];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              float blk[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) blk[i] = hv[32 * b + i];
              sb[b] = mx_quant32(blk, c[b]);
            }
            if (row_ok) {
              const int m = 32 * q + lane;
              uint8_t* sc = p.hsc + (static_cast<size_t>(T.g) * p.KBF + (f0 >> 7)) * 512 +
                            sf_byte(m, (f0 & 127) >> 5);
              *reinterpret_cast<uint16_t*>(sc) = static_cast<uint16_t>(sb[0] | (sb[1] << 8));
            }
            if (vw == 32) {
              if (lane == 0) bulk_wait_read<0>();
              __syncwarp();
              uint4* row = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                row[2 * b] = make_uint4(c[b][0], c[b][1], c[b][2], c[b][3]);
                row[2 * b + 1] = make_uint4(c[b][4], c[b][5], c[b][6], c[b][7]);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&map_o, buf, f0, y);
                bulk_commit();
              }
            } else if (row_ok) {
              uint4* dst = reinterpret_cast<uint4*>(p.hq + r * p.Nout + f0);
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                dst[2 * b] = make_uint4(c[b][0], c[b][1], c[b][2], c[b][3]);
                dst[2 * b + 1] = make_uint4(c[b][4], c[b][5], c[b][6], c[b][7]);
              }
            }
          }
        } else if constexpr (KIND == kKSwigluBwd) {
          if (tma_z) {
            // chunks 2 hh + cc: wait for the slot, dz over z in place, two
            // TMA stores, then (half 0) refill the slot with the chunk two on
            bool ok = true;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {  // unrolled: v is indexed by constants
              const int f = 256 * T.nt + 128 * hh + 64 * cc;
              if (!ok || f >= p.Nout) continue;
              ok = __all_sync(0xffffffffu, mbar_wait(&s.zbar[ew][cc], zpar[cc], wc));
              if (!ok) continue;
              zpar[cc] ^= 1u;
              zout[cc] = false;
              uint8_t* sl = buf + cc * 8192 + lane * 128;
#pragma unroll
              for (int h32 = 0; h32 < 2; ++h32) {
                uint4 zg[4], zu[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int off = ((4 * h32 + i) ^ (lane & 7)) << 4;
                  zg[i] = *reinterpret_cast<const uint4*>(sl + off);
                  zu[i] = *reinterpret_cast<const uint4*>(sl + 4096 + off);
                }
                uint32_t wg[16], wu[16];
                swiglu_bwd32(*reinterpret_cast<const uint32_t(*)[32]>(&v[64 * cc + 32 * h32]), zg, zu,
                             wg, wu);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int off = ((4 * h32 + i) ^ (lane & 7)) << 4;
                  *reinterpret_cast<uint4*>(sl + off) =
                      make_uint4(wg[4 * i], wg[4 * i + 1], wg[4 * i + 2], wg[4 * i + 3]);
                  *reinterpret_cast<uint4*>(sl + 4096 + off) =
                      make_uint4(wu[4 * i], wu[4 * i + 1], wu[4 * i + 2], wu[4 * i + 3]);
                }
              }
              fence_proxy_async_smem();
              __syncwarp();
              const int f2 = f + 128;  // the chunk that reuses this slot
              const bool refill = hh == 0 && f2 < p.Nout;
              if (lane == 0) {
                tma_store_2d(&map_h, buf + cc * 8192, f, y);
                tma_store_2d(&map_h, buf + cc * 8192 + 4096, p.Nout + f, y);
                bulk_commit();
                if (refill) {
                  bulk_wait_read<0>();
                  zload(cc, f2, y);
                }
              }
              zout[cc] = refill;
              __syncwarp();
            }
            if (!ok) {
              aborted = true;
              break;
            }
            continue;
          }
          // a partial warp: dh for f = fb .. fb + 127 of each valid row, z read
          // and dz written by the row's own thread (z and dz are [gate | up] rows)
          if (row_ok) {
            const int fb = 256 * T.nt + 128 * hh;
            const __nv_bfloat16* zr = p.zin + r * 2 * p.Nout;
            __nv_bfloat16* dzr = p.out + r * 2 * p.Nout;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              const int f = fb + 32 * ch;
              if (f >= p.Nout) break;
              uint4 zg[4], zu[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                zg[i] = reinterpret_cast<const uint4*>(zr + f)[i];
                zu[i] = reinterpret_cast<const uint4*>(zr + p.Nout + f)[i];
              }
              uint32_t wg[16], wu[16];
              swiglu_bwd32(*reinterpret_cast<const uint32_t(*)[32]>(&v[32 * ch]), zg, zu, wg, wu);
              uint4* og = reinterpret_cast<uint4*>(dzr + f);
              uint4* ou = reinterpret_cast<uint4*>(dzr + p.Nout + f);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                og[i] = make_uint4(wg[4 * i], wg[4 * i + 1], wg[4 * i + 2], wg[4 * i + 3]);
                ou[i] = make_uint4(wu[4 * i], wu[4 * i + 1], wu[4 * i + 2], wu[4 * i + 3]);
              }
            }
          }
        } else {
          const int d0 = 256 * T.nt + 128 * hh;
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const int col = d0 + 64 * ch;
            if (col >= p.Nout) break;
            uint32_t w0[16], w1[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              w0[i] = pack_bf16x2(__uint_as_float(v[64 * ch + 2 * i]),
                                  __uint_as_float(v[64 * ch + 2 * i + 1]));
              w1[i] = pack_bf16x2(__uint_as_float(v[64 * ch + 32 + 2 * i]),
                                  __uint_as_float(v[64 * ch + 32 + 2 * i + 1]));
            }
            if (vw == 32) {
              if (lane == 0) bulk_wait_read<0>();
              __syncwarp();
              put_half_sw(buf, lane, 0, w0);
              put_half_sw(buf, lane, 1, w1);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&map_o, buf, col, y);
                bulk_commit();
              }
            } else if (row_ok) {
              uint4* dst = reinterpret_cast<uint4*>(p.out + r * p.Nout + col);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w0[4 * i], w0[4 * i + 1], w0[4 * i + 2], w0[4 * i + 3]);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[4 + i] = make_uint4(w1[4 * i], w1[4 * i + 1], w1[4 * i + 2], w1[4 * i + 3]);
            }
          }
        }
      }
    }
    if (lane == 0) {
      for (int c = 0; c < 2; ++c)  // z loads still in flight (after an abort) land first
        if (zout[c]) (void)mbar_wait_drain(&s.zbar[ew][c], zpar[c], 100000000ull);
      bulk_wait_all();  // every store has finished before the CTA exits
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Tensor map, dims innermost first, strides in bytes for dims 1..rank-1.
bool make_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, int rank,
              const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
              CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bd[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bd[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides[i];
  return fn(m, type, rank, const_cast<void*>(base), gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND>
cudaError_t launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                        const CUtensorMap& mz, const CUtensorMap& mh, const MxParams& p,
                        long max_tiles, cudaStream_t s) {
  auto kern = mx_gemm_kernel<KIND>;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(MxCfg<KIND>::kSmemBytes));
    if (err != cudaSuccess) return err;
    attr_set[dev].store(true, std::memory_order_release);
  }
  long grid = sm_count();
  if (max_tiles < grid) grid = max_tiles;
  if (grid <= 0) return cudaSuccess;
  kern<<<static_cast<int>(grid), kThreads, MxCfg<KIND>::kSmemBytes, s>>>(ma, mb, mo, mz, mh, p);
  return cudaGetLastError();
}

template <bool TOKENS>
cudaError_t launch_tq(const TqArgs& a, const CUtensorMap& map_q, long max_items,
                      cudaStream_t s) {
  auto kern = mx_transpose_quantize_kernel<TOKENS>;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTqSmem);
    if (err != cudaSuccess) return err;
    attr_set[dev].store(true, std::memory_order_release);
  }
  long grid = static_cast<long>(kTqCtasPerSm) * sm_count();
  if (max_items < grid) grid = max_items;
  if (grid <= 0) return cudaSuccess;
  kern<<<static_cast<unsigned>(grid), kTqThreads, kTqSmem, s>>>(map_q, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mx_quantize_weights(const uint16_t* w, uint8_t* q, uint8_t* sc, uint8_t* q2,
                                       uint8_t* sc2, int E, int Kd, int N, bool fc1_interleave,
                                       cudaStream_t s) {
  TqArgs a{};
  a.src = w;
  a.q = q;
  a.sc = sc;
  a.q2 = q2;
  a.sc2 = sc2;
  a.C = N;
  a.E = E;
  a.Kd = Kd;
  a.KB = static_cast<int>(mx_kblocks(Kd));
  a.NBp = static_cast<int>(mx_weight_row_blocks(N));
  a.KB2 = static_cast<int>(mx_kblocks(N));
  a.NBp2 = static_cast<int>(mx_weight_row_blocks(Kd));
  a.interleave = fc1_interleave ? 1 : 0;
  CUtensorMap mq{};
  if (q != nullptr) {  // the transposed codes as [E * N rows][Kd], 64-row stores
    const uint64_t dims[2] = {static_cast<uint64_t>(Kd), static_cast<uint64_t>(E) * N};
    const uint64_t str[1] = {static_cast<uint64_t>(Kd)};
    const uint32_t box[2] = {128, 64};
    if (!make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, 2, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const long items = mx_cdiv(N, kTqCols) * a.KB * E;
  return launch_tq<false>(a, mq, items, s);
}

cudaError_t launch_mx_permute_quantize(const uint16_t* x, const int32_t* pos, const int32_t* offs,
                                       uint8_t* xq, uint8_t* xsc, const moe_dims& d,
                                       cudaStream_t s) {
  if (d.T == 0) return cudaSuccess;
  long blocks = mx_cdiv(d.T, kPqWarps);
  const long cap = 8L * sm_count();
  if (blocks > cap) blocks = cap;
  mx_permute_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      x, pos, offs, xq, xsc, d.T, d.D, d.K, d.E, static_cast<int>(mx_kblocks(d.D)));
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_rows(const uint16_t* src, const int32_t* offs, uint8_t* q,
                                    uint8_t* sc, int C, const moe_dims& d, cudaStream_t s) {
  const long R = static_cast<long>(d.T) * d.K;
  if (R == 0) return cudaSuccess;
  long blocks = mx_cdiv(R, kPqWarps);
  const long cap = 8L * sm_count();
  if (blocks > cap) blocks = cap;
  mx_permute_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      src, nullptr, offs, q, sc, static_cast<int>(R), C, 1, d.E,
      static_cast<int>(mx_kblocks(C)));
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_tokens(const uint16_t* src, const int32_t* row_src,
                                      const int32_t* offs, uint8_t* qt, uint8_t* sct, int C,
                                      const moe_dims& d, cudaStream_t s) {
  if (static_cast<long>(d.T) * d.K == 0) return cudaSuccess;
  TqArgs a{};
  a.src = src;
  a.row_src = row_src;
  a.offs = offs;
  a.q = qt;
  a.sc = sct;
  a.Rp = mx_token_cols(d);
  a.C = C;
  a.K = d.K;
  a.E = d.E;
  a.NBp = static_cast<int>(mx_weight_row_blocks(C));
  CUtensorMap mq{};
  const uint64_t dims[2] = {static_cast<uint64_t>(a.Rp), static_cast<uint64_t>(C)};
  const uint64_t str[1] = {static_cast<uint64_t>(a.Rp)};
  const uint32_t box[2] = {128, 64};
  if (!make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qt, 2, dims, str, box,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  return launch_tq<true>(a, mq, mx_cdiv(C, kTqCols) * mx_tile_bound(d), s);
}

cudaError_t launch_mx_grouped_gemm(const MxGemmCall& c, cudaStream_t s) {
  const moe_dims& d = c.d;
  const long R = static_cast<long>(d.T) * d.K;
  if (R == 0) return cudaSuccess;
  MxParams p{};
  p.sfa = c.a_sc;
  p.sfb = c.b_sc;
  p.offs = c.offs;
  p.hq = c.hq;
  p.hsc = c.hsc;
  p.out = reinterpret_cast<__nv_bfloat16*>(c.out);
  p.zin = reinterpret_cast<const __nv_bfloat16*>(c.z_in);
  p.zout = reinterpret_cast<__nv_bfloat16*>(c.z_out);
  p.status = c.dev_status;
  p.limit_ns = kDefaultWaitLimitNs;
  p.E = d.E;
  const long Rp = mx_token_cols(d);
  long Nb = 0;  // B rows per expert
  switch (c.kind) {
    case MxKind::kFc1: p.Kd = d.D; Nb = 2L * d.F; p.Nout = d.F; break;
    case MxKind::kRows: p.Kd = c.kd; Nb = c.n; p.Nout = c.n; break;
    case MxKind::kRowsSwigluBwd: p.Kd = d.D; Nb = d.F; p.Nout = d.F; break;
    case MxKind::kWgrad:
      if (Rp > (1L << 30)) return cudaErrorInvalidValue;
      p.Kd = static_cast<int>(Rp);
      Nb = c.n;
      p.Nout = c.n;
      p.Ma = c.m;
      p.m_tiles = static_cast<int>(mx_cdiv(c.m, 128));
      p.NBpA = static_cast<int>(mx_weight_row_blocks(c.m));
      break;
  }
  p.KB = static_cast<int>(mx_kblocks(p.Kd));
  p.NBp = static_cast<int>(mx_weight_row_blocks(Nb));
  p.n_tiles = static_cast<int>(mx_cdiv(Nb, 256));
  p.KBF = static_cast<int>(mx_kblocks(d.F));
  CUtensorMap ma, mb, mo;
  const uint32_t abox[2] = {128, 128};
  const uint32_t bbox[3] = {128, 256, 1};
  const uint32_t obox[2] = {64, 32};
  bool ok;
  if (c.kind == MxKind::kWgrad) {
    // A [m][Rp], B [n][Rp]: token-axis codes; the k coordinate is the token column
    const uint64_t adims[2] = {static_cast<uint64_t>(Rp), static_cast<uint64_t>(c.m)};
    const uint64_t astr[1] = {static_cast<uint64_t>(Rp)};
    const uint64_t bdims[3] = {static_cast<uint64_t>(Rp), static_cast<uint64_t>(Nb), 1};
    const uint64_t bstr[2] = {static_cast<uint64_t>(Rp), static_cast<uint64_t>(Rp) * Nb};
    ok = make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.a, 2, adims, astr, abox,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.b, 3, bdims, bstr, bbox,
                  CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const uint64_t adims[2] = {static_cast<uint64_t>(p.Kd), static_cast<uint64_t>(R)};
    const uint64_t astr[1] = {static_cast<uint64_t>(p.Kd)};
    const uint64_t bdims[3] = {static_cast<uint64_t>(p.Kd), static_cast<uint64_t>(Nb),
                               static_cast<uint64_t>(d.E)};
    const uint64_t bstr[2] = {static_cast<uint64_t>(p.Kd), static_cast<uint64_t>(p.Kd) * Nb};
    ok = make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.a, 2, adims, astr, abox,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.b, 3, bdims, bstr, bbox,
                  CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return cudaErrorInvalidValue;
  const long max_tiles = c.kind == MxKind::kWgrad
                             ? static_cast<long>(d.E) * p.m_tiles * p.n_tiles
                             : mx_tile_bound(d) * p.n_tiles;
  switch (c.kind) {
    case MxKind::kFc1: {
      // h codes: 32 rows x 64 bytes per store, unswizzled staging (or a dummy
      // map over the bf16 h when only that is written)
      const uint64_t odims[2] = {static_cast<uint64_t>(d.F), static_cast<uint64_t>(R)};
      if (c.hq != nullptr) {
        const uint64_t ostr[1] = {static_cast<uint64_t>(d.F)};
        ok = make_map(&mo, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.hq, 2, odims, ostr, obox,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
      } else {
        const uint64_t ostr[1] = {static_cast<uint64_t>(d.F) * 2};
        ok = make_map(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.out, 2, odims, ostr, obox,
                      CU_TENSOR_MAP_SWIZZLE_128B);
      }
      if (!ok) return cudaErrorInvalidValue;
      // training: z and the bf16 h through TMA stores
      CUtensorMap mz = mo, mh = mo;
      if (c.z_out != nullptr) {
        const uint64_t zdims[2] = {2 * static_cast<uint64_t>(d.F), static_cast<uint64_t>(R)};
        const uint64_t zstr[1] = {static_cast<uint64_t>(d.F) * 4};
        if (!make_map(&mz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.z_out, 2, zdims, zstr, obox,
                      CU_TENSOR_MAP_SWIZZLE_128B))
          return cudaErrorInvalidValue;
      }
      if (c.hq != nullptr && c.out != nullptr) {
        const uint64_t hstr[1] = {static_cast<uint64_t>(d.F) * 2};
        if (!make_map(&mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.out, 2, odims, hstr, obox,
                      CU_TENSOR_MAP_SWIZZLE_128B))
          return cudaErrorInvalidValue;
      }
      return launch_gemm<kKFc1>(ma, mb, mo, mz, mh, p, max_tiles, s);
    }
    case MxKind::kRowsSwigluBwd: {
      // z in and dz out, both [R][2F] bf16, 64-column chunks of 32 rows
      const uint64_t odims[2] = {2 * static_cast<uint64_t>(d.F), static_cast<uint64_t>(R)};
      const uint64_t ostr[1] = {static_cast<uint64_t>(d.F) * 4};
      CUtensorMap mz;
      if (!make_map(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.out, 2, odims, ostr, obox,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
          !make_map(&mz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.z_in, 2, odims, ostr, obox,
                    CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
      return launch_gemm<kKSwigluBwd>(ma, mb, mo, mz, mo, p, max_tiles, s);
    }
    case MxKind::kRows:
    case MxKind::kWgrad: {
      const uint64_t rows = c.kind == MxKind::kWgrad ? static_cast<uint64_t>(d.E) * c.m
                                                      : static_cast<uint64_t>(R);
      const uint64_t odims[2] = {static_cast<uint64_t>(p.Nout), rows};
      const uint64_t ostr[1] = {static_cast<uint64_t>(p.Nout) * 2};
      if (!make_map(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.out, 2, odims, ostr, obox,
                    CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
      if (c.kind == MxKind::kWgrad)
        return launch_gemm<kKWgrad>(ma, mb, mo, mo, mo, p, max_tiles, s);
      return launch_gemm<kKRows>(ma, mb, mo, mo, mo, p, max_tiles, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
