// Grouped GEMMs of the MoE block on the fifth-generation tensor cores.
//
// What is computed (per expert e, rows r of its group):
//   FC1 + SwiGLU  a = xs[r] . wi[e] over the whole prefused wi [E, D, 2F];
//                 h = silu(a[:F]) * a[F:], z = a            (MaxText "Keep fused
//                 MoE weights intact through FSDP gather", Description)
//   FC2           ys[r] = h[r] . wo[e]                      (TransformerEngine
//                 "[DRAFT][JAX] Optimize MoE block", Flowchart)
//   dlhs of FC2   dh[r] = dys[r] . wo[e]^T, with the SwiGLU backward fused
//                 into the epilogue (dz = [dgate | dup] as one tensor, MaxText
//                 "Gemma4 26B MoE on TPU v6e", Commits table row 7)
//   dlhs of FC1   dxs[r] = dz[r] . wi[e]^T                  (the transposed-RHS
//                 backward named under Related PRs of the MaxText fused
//                 permute/combine page)
//   drhs          dwo[e] = h_e^T . dys_e,  dwi[e] = xs_e^T . dz_e
// The grouped GEMM is group-aware: ragged group edges are handled inside the
// kernel (row masks in the epilogue, zero-filled reduction tails), never by a
// separate masking pass (TransformerEngine page, Changes).
//
// Design: persistent warp-specialised kernel, one CTA per SM, 192 threads.
//   warp 0     TMA producer: 128x64 A tiles and (BN/CG)x64 B tiles (bf16,
//              128-byte swizzle) into a shared-memory ring, one box per
//              operand (MN-major operands through a map with a chunk
//              dimension); the per-expert weights come through maps whose
//              outer coordinate is the expert.  For drhs the even CTA's
//              producer also claims tiles for the dynamic schedule.
//   warp 1     TMEM allocation (512 columns: two 128xBN fp32 accumulators,
//              or one 512 wide for drhs pair tiles) and MMA issue: one
//              thread issues tcgen05.mma (K=16) and tcgen05.commit; for drhs
//              the warp zero-fills the rows of the last reduction block that
//              belong to the next group.
//   warps 2-5  epilogue: tcgen05.ld (one row per thread), SwiGLU / SwiGLU
//              backward / bf16 conversion, staged in swizzled shared memory
//              and written by TMA stores; with two accumulators the next
//              tile's MMAs overlap it.
// CG = 2 runs the CTA pair of a 2-CTA cluster on one 256-row tile: each CTA
// loads its own 128 A rows and half of the B columns, the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256) reading both CTAs' shared memory, and
// each CTA's TMEM holds its 128 rows.  Both CTAs' loads complete on the even
// CTA's barrier (TMA with .cta_group::2); commits are multicast to both CTAs.
// This halves the B bytes each SM loads per MMA.
// Tiles are scheduled on the device from group_offsets (no host sync):
// forward/dlhs tiles are (expert, 128*CG-row block, N block) with the rows of
// a block starting at the group's first row; drhs tiles are (expert, M
// block, N block) with the group's rows as the reduction.
#include <cuda.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kUmmaK = 16;
constexpr int kAStageBytes = BM * BK * 2;  // 16 KB
constexpr int kChunkBytes = 64 * BK * 2;   // one 64-wide MN chunk of 64 K rows: 8 KB
constexpr int kThreads = 192;
constexpr int kMaxExperts = 1024;
constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 4;
constexpr int kBufBytes = 32 * 128;  // staging buffer: 32 rows x 64 bf16
constexpr size_t kSmemLimit = 227 * 1024;
constexpr int kSched = 8;  // tile-index slots of the dynamic (drhs) schedule

// CAP: experts the offset and block-prefix arrays hold (the launch's E must
// not exceed it).
template <int CAP>
struct SmemCtlT {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t zbar[kEpiWarps][2];  // z rows landed in a slot of an epilogue warp
  uint64_t sfull[kSched];    // a tile index was written to the slot
  uint64_t sempty[kSched];   // every role has read the slot
  int sched[kSched];
  uint32_t tmem_base;
  int abort_flag;
  int off[CAP + 1];  // group offsets
  // forward/dlhs: prefix of (128*CG)-row blocks per group; drhs: sort keys
  // whose low 10 bits are the experts by descending reduction length
  int mt[CAP + 1];
};
using SmemCtl = SmemCtlT<kMaxExperts>;

// Tile shape: 128 x BN accumulator per CTA, CG CTAs per MMA, a `STAGES`-deep
// operand ring, RING staging buffers per epilogue warp, and (ZB > 0) ZB slots
// per epilogue warp into which TMA loads the z rows that the fused SwiGLU
// backward reads and from which it stores dz (no staging ring needed then).
// A z slot holds the gate and up halves of 32 rows x ZW columns: 8 KB at 64
// columns (128-byte rows), 4 KB at 32 (64-byte rows, 64-byte swizzle).
//
// NACC = 2 makes a tile two accumulators wide (2*BN columns per CTA, all 512
// TMEM columns): each A stage feeds two MMAs, so each SM loads 25% fewer bytes
// per MMA, at the price of single-buffered accumulators.
template <int BN_, int STAGES_, int CG_, int RING_, int ZB_ = 0, int NACC_ = 1,
          int MAXE_ = kMaxExperts, int ZW_ = 64>
struct Shape {
  using Ctl = SmemCtlT<MAXE_>;
  static constexpr int kMaxE = MAXE_;
  static constexpr int BN = BN_;
  static constexpr int kStages = STAGES_;
  static constexpr int CG = CG_;
  static constexpr int kRing = RING_;
  static constexpr bool kZB = ZB_ != 0;
  static constexpr int kZSlots = ZB_;
  static constexpr int kNacc = NACC_;
  static constexpr int kZW = ZW_;                  // z chunk width (columns)
  static constexpr int kZBuf = 32 * ZW_ * 2;       // one half (gate or up) of a slot
  static constexpr int kZBytes = kEpiWarps * ZB_ * 2 * kZBuf;
  static constexpr int kBRows = BN / CG;  // B columns held by one CTA, per accumulator
  static constexpr int kBStageBytes = NACC_ * kBRows * BK * 2;
  static constexpr int kStageBytes = kAStageBytes + kBStageBytes;
  static constexpr int kAccSlots = NACC_ == 1 ? 2 : 1;   // double-buffered when 1 wide
  static constexpr int kAccStride = BN * NACC_;           // TMEM columns per slot
  static constexpr int kTmemCols = kAccSlots * kAccStride;
  static_assert(kTmemCols == 512, "TMEM columns");
  static constexpr int kEpiBytes = kEpiWarps * RING_ * kBufBytes;
  static constexpr size_t kSmemBytes =
      1024 + static_cast<size_t>(STAGES_) * kStageBytes + kEpiBytes + kZBytes + sizeof(Ctl);
  static_assert(BN == 256, "tile width");
  static_assert(CG == 1 || CG == 2, "CTA group");
  static_assert(STAGES_ >= 2 && STAGES_ <= kMaxStages, "stages");
  static_assert(RING_ >= (ZB_ ? 0 : 1) && RING_ <= 4, "staging ring");
  static_assert(ZB_ == 0 || ZB_ == 2, "z slots");
  static_assert(ZW_ == 64 || ZW_ == 32, "z chunk width");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory");
};

struct Params {
  const int32_t* offs;
  __nv_bfloat16* out0;
  __nv_bfloat16* out1;
  const __nv_bfloat16* aux;
  int32_t* status;
  unsigned int* tile_ctr;  // drhs: tiles claimed so far (zero at launch)
  const int32_t* row_src;  // gathered FC1, combined FC2: slot j = t*K + k of each row
  const float* wts;        // combined FC2: routing weights [T, K]
  float* acc;              // combined FC2: fp32 [T, D] accumulator
  int Ktop;                // top_k
  int evict_weights;       // weight loads marked L2::evict_first (read once)
  long R;                  // rows (T * K)
  uint64_t limit_ns;
  int E, Kdim, M, N, F;
  int m_tiles, n_tiles;
};

// The kinds that share FC1's (FC2's) operands, tiles and epilogue: the
// gathered FC1 differs only in where its A rows come from, the combined FC2
// only in where its output goes.
template <int KIND>
__host__ __device__ constexpr bool fc1_like() {
  return KIND == static_cast<int>(GemmKind::kFc1) || KIND == static_cast<int>(GemmKind::kFc1Gather);
}
template <int KIND>
__host__ __device__ constexpr bool fc2_like() {
  return KIND == static_cast<int>(GemmKind::kFc2) || KIND == static_cast<int>(GemmKind::kFc2Combine);
}

template <int KIND, int BN, int CG>
struct Traits {
  static constexpr bool kGroupedK = (KIND == static_cast<int>(GemmKind::kDrhsFc2) ||
                                     KIND == static_cast<int>(GemmKind::kDrhsFc1));
  static constexpr bool kAMn = kGroupedK;
  static constexpr bool kBMn = (fc1_like<KIND>() || fc2_like<KIND>() || kGroupedK);
  static constexpr uint32_t kIdesc = instr_desc_bf16(BM * CG, BN, kAMn, kBMn);
};

struct Tile {
  int e;
  int row0;   // this CTA's first output row (forward/dlhs) or first group row (drhs)
  int rows;   // valid rows of this CTA's part of the tile (forward/dlhs)
  int m0;     // drhs: this CTA's first output row (of F or D)
  int n0;     // first output column of the tile
  int kb;     // reduction blocks of 64
  int klen;   // drhs: group rows
};

template <int KIND, int BN, int CG, class Ctl>
__device__ __forceinline__ Tile decode_tile(int t, int rank, const Params& p, const Ctl& s) {
  Tile T;
  if constexpr (!Traits<KIND, BN, CG>::kGroupedK) {
    const int mt = t / p.n_tiles;
    const int nt = t - mt * p.n_tiles;
    int lo = 0, hi = p.E - 1;  // largest e with mt[e] <= mt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s.mt[mid] <= mt) lo = mid;
      else hi = mid - 1;
    }
    T.e = lo;
    T.row0 = s.off[lo] + (mt - s.mt[lo]) * (BM * CG) + BM * rank;
    T.rows = max(0, min(BM, s.off[lo + 1] - T.row0));
    T.m0 = 0;
    T.n0 = nt * (fc1_like<KIND>() ? BN / 2 : BN);
    T.kb = p.Kdim / BK;
    T.klen = p.Kdim;
  } else {
    const int per_e = p.m_tiles * p.n_tiles;
    const int i = t / per_e;
    T.e = s.mt[i] & (kMaxExperts - 1);
    const int r = t - i * per_e;
    const int mt = r / p.n_tiles;
    T.m0 = mt * (BM * CG) + BM * rank;
    T.n0 = (r - mt * p.n_tiles) * BN;
    T.row0 = s.off[T.e];
    T.klen = s.off[T.e + 1] - T.row0;
    T.rows = BM;
    T.kb = (T.klen + BK - 1) / BK;
  }
  return T;
}

template <int KIND, int BN, int CG, class Ctl>
__device__ __forceinline__ int total_tiles(const Params& p, const Ctl& s) {
  if constexpr (!Traits<KIND, BN, CG>::kGroupedK) return s.mt[p.E] * p.n_tiles;
  else return p.E * p.m_tiles * p.n_tiles;
}

// Dynamic tile schedule of the drhs GEMMs.  Their tiles take as long as
// their group has rows, so a fixed assignment leaves pairs idle while
// others finish long groups.  Instead the even CTA's producer claims tile
// indices from a global counter, in the order of descending group length
// (longest first, so that the last tiles handed out are the short ones), and
// writes each index into one of kSched shared-memory slots of both CTAs; the
// MMA warp, the epilogue warps and the odd CTA's producer read it from there
// and release the slot on the even CTA's `sempty` barrier.  An index >=
// the tile count ends the sequence.

// Readers of one slot: the MMA warp and the epilogue warps of the even CTA,
// plus the producer and the epilogue warps of the odd CTA.
template <int CG>
__host__ __device__ constexpr uint32_t sched_readers() { return CG == 2 ? 2 * kEpiWarps + 2 : kEpiWarps + 1; }

// Next tile index for a reader (every thread of `mask` calls it; `releaser`
// releases the slot).  Returns -1 when the wait gave up.
template <int CG, class Ctl>
__device__ __forceinline__ int sched_take(Ctl& s, uint32_t& seq, bool leader, bool releaser,
                                          unsigned mask, const WaitCtl& wc) {
  const uint32_t slot = seq % kSched;
  const uint32_t par = (seq / kSched) & 1u;
  ++seq;
  const bool got = (CG == 2) ? mbar_wait_cluster(&s.sfull[slot], par, wc)
                             : mbar_wait(&s.sfull[slot], par, wc);
  if (!__all_sync(mask, got)) return -1;
  const int t = *reinterpret_cast<volatile int*>(&s.sched[slot]);
  __syncwarp(mask);
  if (releaser) {
    if (CG == 2 && !leader)
      mbar_arrive_remote(mapa_shared(smem_u32(&s.sempty[slot]), 0));
    else
      mbar_arrive(&s.sempty[slot]);
  }
  return t;
}

// The even CTA's producer publishes tile index t to every reader.  Returns
// false when the wait for a free slot gave up.
template <int CG, class Ctl>
__device__ __forceinline__ bool sched_publish(Ctl& s, uint32_t& seq, int t, const WaitCtl& wc) {
  const uint32_t slot = seq % kSched;
  const uint32_t par = (seq / kSched) & 1u;
  ++seq;
  const bool free_slot = (CG == 2) ? mbar_wait_cluster(&s.sempty[slot], par ^ 1u, wc)
                                   : mbar_wait(&s.sempty[slot], par ^ 1u, wc);
  if (!free_slot) return false;
  *reinterpret_cast<volatile int*>(&s.sched[slot]) = t;
  if constexpr (CG == 2) {
    st_cluster_u32(mapa_shared(smem_u32(&s.sched[slot]), 1), static_cast<uint32_t>(t));
    mbar_arrive_remote(mapa_shared(smem_u32(&s.sfull[slot]), 1));
  }
  mbar_arrive(&s.sfull[slot]);
  return true;
}

// Orders the experts by descending reduction length (64-row blocks; ties by
// expert index) into s.mt, identically in every CTA: bitonic sort of
// 32-bit keys (blocks, clamped to 22 bits, inverted | expert).  All threads
// of the CTA call it after s.off is complete.
template <class Ctl>
__device__ __forceinline__ void sort_groups_desc(Ctl& s, int E) {
  int n = 1;
  while (n < E) n <<= 1;
  uint32_t* key = reinterpret_cast<uint32_t*>(s.mt);
  for (int i = threadIdx.x; i < n; i += kThreads) {
    uint32_t k = 0xFFFFFFFFu;
    if (i < E) {
      const int kb = min((s.off[i + 1] - s.off[i] + BK - 1) / BK, 0x3FFFFF);
      k = (static_cast<uint32_t>(0x3FFFFF - kb) << 10) | static_cast<uint32_t>(i);
    }
    key[i] = k;
  }
  __syncthreads();
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int l = i ^ j;
        if (l > i) {
          const uint32_t a = key[i], b = key[l];
          if ((a > b) == ((i & k) == 0)) {
            key[i] = b;
            key[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// How many of the first n uses of a ring of S slots (taken in order 0, 1,
// ..., S-1, 0, ...) fell on slot i.  The producer and MMA loops keep one
// count instead of a per-slot array (which a run-time index would put in
// local memory).
__device__ __forceinline__ uint32_t ring_uses(uint32_t n, uint32_t i, uint32_t S) {
  return n > i ? (n - i + S - 1) / S : 0u;
}

// One TMA load of a stage: for a pair, the bytes complete on the even CTA's
// barrier (`bar` is then its shared::cluster address).
template <int CG>
__device__ __forceinline__ void load2(void* dst, const CUtensorMap* map, uint32_t bar, int c0,
                                      int c1) {
  if constexpr (CG == 1) tma_load_2d_addr(dst, map, bar, c0, c1);
  else tma_load_2d_pair(dst, map, bar, c0, c1);
}
template <int CG>
__device__ __forceinline__ void load3(void* dst, const CUtensorMap* map, uint32_t bar, int c0,
                                      int c1, int c2) {
  if constexpr (CG == 1) tma_load_3d_addr(dst, map, bar, c0, c1, c2);
  else tma_load_3d_pair(dst, map, bar, c0, c1, c2);
}
template <int CG>
__device__ __forceinline__ void load4(void* dst, const CUtensorMap* map, uint32_t bar, int c0,
                                      int c1, int c2, int c3) {
  if constexpr (CG == 1) tma_load_4d_addr(dst, map, bar, c0, c1, c2, c3);
  else tma_load_4d_pair(dst, map, bar, c0, c1, c2, c3);
}

// Four rows of a 2-D map whose box is 64 columns x 1 row, gathered into 512
// consecutive bytes of shared memory (four 128-byte rows, swizzled by their
// shared-memory address like any tile).
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int r0, int r1, int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}

// L2 policy of the expert-weight loads.  Where groups average at most one
// lone-CTA row block, each weight byte is read once per GEMM; the loads are
// then marked to leave L2 first (L2::evict_first), which keeps the
// activations the step re-reads (xs across N tiles, ys for the combine) in
// L2 (1024 tokens, E = 128: combine 12.2 -> 10.2 us, FC1 155 -> 151 us).
// With larger groups row blocks of one expert re-read its weights, and the
// hint costs more than it saves (8192 tokens: FC2 175 -> 183 us), so the
// loads keep the normal policy.
// (Not volatile: a kind that loads no weights drops it.)
__device__ __forceinline__ uint64_t weight_policy(int evict_first) {
  uint64_t pol;
  if (evict_first)
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  else
    asm("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
template <int CG>
__device__ __forceinline__ void load3w(void* dst, const CUtensorMap* map, uint32_t bar, int c0,
                                       int c1, int c2, uint64_t pol) {
  if constexpr (CG == 1)
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2.L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
        : "memory");
}
template <int CG>
__device__ __forceinline__ void load4w(void* dst, const CUtensorMap* map, uint32_t bar, int c0,
                                       int c1, int c2, int c3, uint64_t pol) {
  if constexpr (CG == 1)
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "l"(pol)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2.L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "l"(pol)
        : "memory");
}

// MMA width of accumulator `a` of tile T: its valid output columns rounded
// up to what the B layout allows (whole 64-column chunks per CTA for an
// MN-major B, 8-row groups per CTA for a K-major B); 0 when the accumulator
// lies wholly past the last column.  Narrow tail tiles thus cost only their
// valid columns.  For FC1 the width is that of gate and up together:
// columns [0, w/2) are gate columns n0.., [w/2, w) up columns F + n0...
template <int KIND, int BN, int CG>
__device__ __forceinline__ int acc_cols(const Tile& T, int a, const Params& p) {
  if constexpr (fc1_like<KIND>()) {
    return 2 * min(BN / 2, p.N - T.n0);  // p.N = F, a multiple of 64
  } else {
    const int nv = min(BN, p.N - (T.n0 + a * BN));
    if (nv <= 0) return 0;
    constexpr int g = Traits<KIND, BN, CG>::kBMn ? 64 * CG : 16 * CG;
    return min(BN, (nv + g - 1) / g * g);
  }
}

// Whether accumulator `a` of T is narrower than a full tile in a kind whose B
// columns, when narrow, come in single 64-wide chunks (the multi-chunk box
// would put them at the wrong offsets of a pair's halves).
template <int KIND, int BN, int CG>
__device__ __forceinline__ bool narrow_chunks(int w) {
  return (fc2_like<KIND>() || Traits<KIND, BN, CG>::kGroupedK) && w < BN;
}

// Bytes that one reduction block of tile T brings into ONE CTA's stage.
template <int KIND, int BN, int CG, int NACC>
__device__ __forceinline__ uint32_t stage_bytes(const Tile& T, const Params& p) {
  constexpr int kBChunks = BN / 64 / CG;
  if constexpr (KIND == static_cast<int>(GemmKind::kDlhsFc2) ||
                KIND == static_cast<int>(GemmKind::kDlhsFc1)) {
    return kAStageBytes + (BN / CG) * BK * 2;  // K-major B: one box of BN/CG rows
  } else if constexpr (fc1_like<KIND>()) {
    return kAStageBytes + kBChunks * kChunkBytes;  // whole boxes, also for the tail
  } else {
    uint32_t chunks = 0;
#pragma unroll
    for (int a = 0; a < NACC; ++a) {
      const int w = acc_cols<KIND, BN, CG>(T, a, p);
      chunks += narrow_chunks<KIND, BN, CG>(w) ? w / (64 * CG) : kBChunks;
    }
    return kAStageBytes + chunks * kChunkBytes;
  }
}

// TMA loads of one reduction block: this CTA's 128 A rows and its share of
// the B columns: of an accumulator w columns wide, CTA `rank` of a pair
// holds columns [rank*w/2, (rank+1)*w/2), which tcgen05.mma.cta_group::2
// takes as accumulator columns in that order.  An MN-major operand's 64-wide
// chunks come in ONE box per operand and accumulator (a map with a chunk
// dimension of stride 128 bytes): the number of TMA instructions, more than
// their bytes, limits how fast a stage fills.  Maps: A (map_a), B (map_b),
// and for narrow fc2/drhs accumulators B in single chunks (map_d).
template <int KIND, int BN, int CG, int NACC = 1>
__device__ __forceinline__ void issue_loads(const Tile& T, int kb, int rank, uint8_t* sa,
                                            uint8_t* sb, uint32_t bar, const CUtensorMap* ma,
                                            const CUtensorMap* mb, const CUtensorMap* md,
                                            const Params& p) {
  const int k0 = kb * BK;
  constexpr int kBChunks = BN / 64 / CG;  // 64-wide B chunks a CTA holds per accumulator
  const uint64_t wpol = weight_policy(p.evict_weights);
  if constexpr (fc1_like<KIND>()) {
    // B = wi[e] as [chunk of 2F][D][64]: for a pair the even CTA takes the
    // gate chunks n0.., the odd one the up chunks F + n0..; alone, a CTA
    // takes both (gate in slots [0, kBChunks/2), up after).  The gathered
    // FC1's A rows are copied by the producer warp instead.
    if constexpr (KIND != static_cast<int>(GemmKind::kFc1Gather)) load2<CG>(sa, ma, bar, k0, T.row0);
    if constexpr (CG == 1) {
      load4w<CG>(sb, mb, bar, 0, k0, T.n0 / 64, T.e, wpol);
      load4w<CG>(sb + (kBChunks / 2) * kChunkBytes, mb, bar, 0, k0, (p.F + T.n0) / 64, T.e, wpol);
    } else {
      load4w<CG>(sb, mb, bar, 0, k0, (rank == 0 ? T.n0 : p.F + T.n0) / 64, T.e, wpol);
    }
  } else if constexpr (fc2_like<KIND>()) {
    const int w = acc_cols<KIND, BN, CG>(T, 0, p);
    load2<CG>(sa, ma, bar, k0, T.row0);
    if (!narrow_chunks<KIND, BN, CG>(w)) {
      load4w<CG>(sb, mb, bar, 0, k0, (T.n0 + (BN / CG) * rank) / 64, T.e, wpol);
    } else {
      for (int j = 0; j < w / (64 * CG); ++j)
        load3w<CG>(sb + j * kChunkBytes, md, bar, T.n0 + (w / CG) * rank + 64 * j, k0, T.e, wpol);
    }
  } else if constexpr (KIND == static_cast<int>(GemmKind::kDlhsFc2) ||
                       KIND == static_cast<int>(GemmKind::kDlhsFc1)) {
    const int w = acc_cols<KIND, BN, CG>(T, 0, p);
    load2<CG>(sa, ma, bar, k0, T.row0);
    load3w<CG>(sb, mb, bar, k0, T.n0 + (w / CG) * rank, T.e, wpol);  // K-major B rows
  } else {
    // A = [chunk of M][R][64], B = [chunk of N][R][64]
    const int kr = T.row0 + k0;
    load3<CG>(sa, ma, bar, 0, kr, T.m0 / 64);
#pragma unroll
    for (int a = 0; a < NACC; ++a) {
      const int w = acc_cols<KIND, BN, CG>(T, a, p);
      uint8_t* sba = sb + a * kBChunks * kChunkBytes;
      if (!narrow_chunks<KIND, BN, CG>(w)) {
        load3<CG>(sba, mb, bar, 0, kr, (T.n0 + a * BN + (BN / CG) * rank) / 64);
      } else {
        for (int j = 0; j < w / (64 * CG); ++j)
          load2<CG>(sba + j * kChunkBytes, md, bar, T.n0 + a * BN + (w / CG) * rank + 64 * j, kr);
      }
    }
  }
}

// The last reduction block of a drhs tile holds `valid` rows of the group
// (1..63); the rest belong to the next group (or lie past the end).  Its MMA
// K-steps of 16 rows that lie wholly past `valid` are skipped; only the rows
// [valid, roundup16(valid)) of the step that straddles the end are zeroed, in
// A and B.  For a pair the even CTA's MMA warp zeroes both CTAs' stages (the
// odd CTA's through the cluster's shared window), since the odd CTA never
// learns when its bytes have landed.
template <int BN, int CG, int NACC = 1>
__device__ __forceinline__ void zero_tail(uint8_t* sa, uint8_t* sb, int valid, int lane) {
  const int end = (valid + kUmmaK - 1) / kUmmaK * kUmmaK;
  const int nrows = end - valid;
  if (nrows == 0) return;
  constexpr int kChunksAB = 2 + NACC * BN / 64 / CG;
  // lane i: 16-byte piece i % 8 of row valid + i / 8, in every 64-wide chunk
  for (int i = lane; i < nrows * 8; i += 32) {
    const int off = (valid + (i >> 3)) * 128 + (i & 7) * 16;
#pragma unroll
    for (int c = 0; c < kChunksAB; ++c) {
      uint8_t* addr = (c < 2 ? sa + c * kChunkBytes : sb + (c - 2) * kChunkBytes) + off;
      *reinterpret_cast<uint4*>(addr) = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (CG == 2) st_cluster_zero16(mapa_shared(smem_u32(addr), 1));
    }
  }
  if constexpr (CG == 2) fence_proxy_async_cluster();
  else fence_proxy_async_smem();
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// ---------------------------------------------------------------- epilogue
// Each epilogue warp owns 32 accumulator rows (its TMEM lane quarter) and a
// ring of staging buffers of 32 rows x 64 bf16 (128-byte rows, 128-byte
// swizzle).  A 64-column slice of its rows is converted, written to a buffer
// (lane = row) and sent to global memory by one TMA bulk-tensor store; the
// store engine writes whole lines, asynchronously.  A warp whose rows
// straddle the end of a group (forward/dlhs only) stores its valid rows with
// per-thread stores instead, so that no row of the next group is touched.
template <int RING>
struct Ring {
  uint8_t* base;
  uint32_t next;

  // Take `n` consecutive buffers; the stores that last read them are done.
  template <int N>
  __device__ __forceinline__ uint8_t* take(int lane) {
    static_assert(N >= 1 && N <= RING, "ring");
    if (lane == 0) bulk_wait_read<RING - N>();
    __syncwarp();
    uint8_t* b = base + (next % RING) * kBufBytes;
    next += N;
    return b;
  }
  __device__ __forceinline__ uint8_t* after(uint8_t* first, int i) const {
    const uint32_t idx = static_cast<uint32_t>((first - base) / kBufBytes + i) % RING;
    return base + idx * kBufBytes;
  }
};

// 16 packed bf16 pairs = 32 columns (half `h` of a 64-column row) of row `lane`.
__device__ __forceinline__ void put_half(uint8_t* buf, int lane, int h, const uint32_t (&w)[16]) {
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int unit = h * 4 + j;
    *reinterpret_cast<uint4*>(row + ((unit ^ (lane & 7)) << 4)) =
        make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

// A buffer of 64-byte rows under the 64-byte swizzle: 16-byte unit j of row
// r sits at unit j ^ ((r >> 1) & 3) of the row (address bits 4-5 XOR bits 7-8).
__device__ __forceinline__ int row64_unit(int r, int j) { return r * 64 + ((j ^ ((r >> 1) & 3)) << 4); }
// 16 packed bf16 pairs = the 32 columns of row `lane` of such a buffer.
__device__ __forceinline__ void put_row64(uint8_t* buf, int lane, const uint32_t (&w)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(buf + row64_unit(lane, j)) =
        make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

__device__ __forceinline__ void pack16(const uint32_t (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    w[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
}

__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&w)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// Make the staged rows visible to the TMA engine (all lanes), then one lane
// stores buffers.
__device__ __forceinline__ void publish() {
  fence_proxy_async_smem();
  __syncwarp();
}
__device__ __forceinline__ void flush_2d(uint8_t* buf, const CUtensorMap* map, int x, int y, int lane) {
  if (lane == 0) {
    tma_store_2d(map, buf, x, y);
    bulk_commit();
  }
}
__device__ __forceinline__ void flush_3d(uint8_t* buf, const CUtensorMap* map, int x, int y, int z,
                                         int lane) {
  if (lane == 0) {
    tma_store_3d(map, buf, x, y, z);
    bulk_commit();
  }
}

// z rows of the fused SwiGLU backward, by TMA: two slots per epilogue warp,
// each the gate and up rows (32 x ZW bf16 each) of one ZW-column chunk.  The
// backward of a chunk is written over the z it read, and stored from there.
// Requests run up to two chunks ahead, into the next tile of the warp's
// (static) schedule: that tile's first chunks then arrive while its
// accumulator is still being computed, instead of one DRAM round trip per
// chunk in the epilogue.
struct ZPipe {
  uint8_t* buf;    // this warp's two slots
  uint64_t* bar;   // their barriers
  uint32_t ph;     // phase bit of each slot
  int send, recv;  // slot of the next request, of the next chunk to consume
  int out;         // requests not yet consumed
  int qt, qch;     // next chunk to request: tile index and chunk
};

template <int RING>
struct EpiCtx {
  const CUtensorMap* map_c;  // out0
  const CUtensorMap* map_d;  // out1 (z of FC1), or z (input of the fused SwiGLU backward)
  Ring<RING> ring;
  int q;                     // lane quarter: rows [32q, 32q+32) of this CTA's tile
  int lane;
  ZPipe zp;
  const WaitCtl* wc;
};

// Whether this warp's z rows come by TMA: the fused SwiGLU backward, a shape
// with z slots, and all 32 of the warp's rows inside the group.
template <int KIND, bool ZB, int RING>
__device__ __forceinline__ bool z_by_tma(const Tile& T, const EpiCtx<RING>& c, const Params& p) {
  return KIND == static_cast<int>(GemmKind::kDlhsFc2) && ZB && p.aux != nullptr &&
         T.rows - 32 * c.q >= 32;
}
// ZW-column chunks of tile T that hold output columns (FC2 dlhs: N = F).
template <int ZW>
__device__ __forceinline__ int z_chunks(const Tile& T, int BN, const Params& p) {
  return max(0, min(BN, p.F - T.n0) + ZW - 1) / ZW;
}
// Request the gate and up z rows of chunk `ch` of tile T into the next slot,
// once the store that last read that slot has read it.
template <int ZW, int RING>
__device__ __forceinline__ void z_issue(const Tile& T, int ch, EpiCtx<RING>& c) {
  constexpr int kZBuf = 32 * ZW * 2;
  ZPipe& z = c.zp;
  if (c.lane == 0) {
    bulk_wait_read<0>();
    uint64_t* b = z.bar + z.send;
    mbar_arrive_expect_tx(b, 2 * kZBuf);
    tma_load_3d_addr(z.buf + z.send * 2 * kZBuf, c.map_d, smem_u32(b), T.n0 + ZW * ch,
                     T.row0 + 32 * c.q, 0);  // gate chunk, then up chunk
  }
  __syncwarp();
  z.send ^= 1;
  ++z.out;
}
// Keep two requests in flight: the rest of tile t's chunks, then (when it
// also takes its z by TMA) the first chunks of the warp's next tile tn.
template <int KIND, int BN, bool ZB, int RING, int ZW>
__device__ __forceinline__ void z_fill(int t, const Tile& T, int tn, const Tile& Tn,
                                       EpiCtx<RING>& c, const Params& p) {
  ZPipe& z = c.zp;
  while (z.out < 2) {
    if (z.qt == t && z.qch < z_chunks<ZW>(T, BN, p)) {
      z_issue<ZW>(T, z.qch++, c);
    } else if (z.qt == t && tn >= 0 && z_by_tma<KIND, ZB, RING>(Tn, c, p)) {
      z.qt = tn;
      z.qch = 0;
    } else if (z.qt == tn && tn >= 0 && z.qch < z_chunks<ZW>(Tn, BN, p)) {
      z_issue<ZW>(Tn, z.qch++, c);
    } else {
      break;
    }
  }
}
// Wait for the oldest request; returns its slot, or -1 when the wait gave up.
template <int RING>
__device__ __forceinline__ int z_take(EpiCtx<RING>& c) {
  ZPipe& z = c.zp;
  const int slot = z.recv;
  if (!mbar_wait(z.bar + slot, (z.ph >> slot) & 1u, *c.wc)) return -1;
  z.ph ^= 1u << slot;
  z.recv ^= 1;
  --z.out;
  return slot;
}
// Requests still in flight land before the CTA exits (bounded).
template <int RING>
__device__ __forceinline__ void z_drain(EpiCtx<RING>& c) {
  ZPipe& z = c.zp;
  while (z.out > 0) {
    (void)mbar_wait_drain(z.bar + z.recv, (z.ph >> z.recv) & 1u, 100000000ull);
    z.ph ^= 1u << z.recv;
    z.recv ^= 1;
    --z.out;
  }
}

// t, tn, Tn: the tile's index and the warp's next tile (index, or -1), for
// the z requests of the fused SwiGLU backward.
template <int KIND, int BN, int CG, int RING, bool ZB, int ZW>
__device__ __forceinline__ void epilogue_tile(const Tile& T, uint32_t tbase, EpiCtx<RING>& c,
                                              const Params& p, int t, int tn, const Tile& Tn) {
  const int lane = c.lane;
  uint32_t v[32];
  uint32_t w[16];
  if constexpr (Traits<KIND, BN, CG>::kGroupedK) {
    // weight gradient tile: rows m0+32q.. of expert e; rows >= M are clipped by the 3-D map
    const int y = T.m0 + 32 * c.q;
    if (y >= p.M) return;
    for (int ch = 0; ch < BN / 64; ++ch) {
      const int col = T.n0 + 64 * ch;
      if (col >= p.N) break;
      uint8_t* buf = c.ring.template take<1>(lane);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmem_ld_32x32b_x32(tbase + 64 * ch + 32 * h, v);
        tmem_ld_wait();
        pack16(v, w);
        put_half(buf, lane, h, w);
      }
      publish();
      flush_3d(buf, c.map_c, col, y, T.e, lane);
    }
  } else {
    const int vw = min(32, max(0, T.rows - 32 * c.q));  // valid rows of this warp
    if (vw == 0) return;
    const bool full = (vw == 32);
    const bool row_ok = lane < vw;
    const int y = T.row0 + 32 * c.q;
    const long r = static_cast<long>(y) + lane;
    if constexpr (fc1_like<KIND>()) {
      const bool with_z = p.out1 != nullptr;
      const int hw = acc_cols<KIND, BN, CG>(T, 0, p) / 2;  // first up column of the accumulator
      for (int ch = 0; ch < BN / 128; ++ch) {
        const int f0 = T.n0 + 64 * ch;
        if (f0 >= p.F) break;
        uint8_t* hb = nullptr;
        if (full) hb = with_z ? c.ring.template take<3>(lane) : c.ring.template take<1>(lane);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t u[32];
          tmem_ld_32x32b_x32(tbase + 64 * ch + 32 * h, v);
          tmem_ld_32x32b_x32(tbase + hw + 64 * ch + 32 * h, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h0 = silu_f(__uint_as_float(v[2 * i])) * __uint_as_float(u[2 * i]);
            const float h1 = silu_f(__uint_as_float(v[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
            w[i] = pack_bf16x2(h0, h1);
          }
          uint32_t wg[16], wu[16];
          if (with_z) {
            pack16(v, wg);
            pack16(u, wu);
          }
          if (full) {
            put_half(hb, lane, h, w);
            if (with_z) {
              put_half(c.ring.after(hb, 1), lane, h, wg);
              put_half(c.ring.after(hb, 2), lane, h, wu);
            }
          } else if (row_ok) {
            store_row32(p.out0 + r * p.F + f0 + 32 * h, w);
            if (with_z) {
              store_row32(p.out1 + r * 2 * p.F + f0 + 32 * h, wg);
              store_row32(p.out1 + r * 2 * p.F + p.F + f0 + 32 * h, wu);
            }
          }
        }
        if (full) {
          publish();
          flush_2d(hb, c.map_c, f0, y, lane);
          if (with_z) flush_3d(c.ring.after(hb, 1), c.map_d, f0, y, 0, lane);  // zg, zu
        }
      }
    } else if constexpr (KIND == static_cast<int>(GemmKind::kDlhsFc2) && ZB) {
      // fused SwiGLU backward on a shape with z slots (these run nothing else)
      if (full) {
        constexpr int kZBuf = 32 * ZW * 2;
        for (int ch = 0; ch < BN / ZW; ++ch) {
          const int f0 = T.n0 + ZW * ch;
          if (f0 >= p.F) break;
          const int slot = z_take(c);
          if (slot < 0) return;
          uint8_t* gbuf = c.zp.buf + slot * 2 * kZBuf;
          uint8_t* ubuf = gbuf + kZBuf;
          if constexpr (ZW == 64) {
            uint4 zg[8], zu[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int off = lane * 128 + ((j ^ (lane & 7)) << 4);
              zg[j] = *reinterpret_cast<const uint4*>(gbuf + off);
              zu[j] = *reinterpret_cast<const uint4*>(ubuf + off);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              tmem_ld_32x32b_x32(tbase + 64 * ch + 32 * h, v);
              tmem_ld_wait();
              uint32_t wg[16], wu[16];
              swiglu_bwd32(v, zg + 4 * h, zu + 4 * h, wg, wu);
              // each lane overwrites its own row of the z it has read
              put_half(gbuf, lane, h, wg);
              put_half(ubuf, lane, h, wu);
            }
          } else {
            uint4 zg[4], zu[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int off = row64_unit(lane, j);
              zg[j] = *reinterpret_cast<const uint4*>(gbuf + off);
              zu[j] = *reinterpret_cast<const uint4*>(ubuf + off);
            }
            tmem_ld_32x32b_x32(tbase + 32 * ch, v);
            tmem_ld_wait();
            uint32_t wg[16], wu[16];
            swiglu_bwd32(v, zg, zu, wg, wu);
            put_row64(gbuf, lane, wg);
            put_row64(ubuf, lane, wu);
          }
          publish();
          flush_3d(gbuf, c.map_c, f0, y, 0, lane);  // dgate, dup
          z_fill<KIND, BN, ZB, RING, ZW>(t, T, tn, Tn, c, p);
        }
        return;
      }
      // a warp with rows past the group's end: z and dz per thread
      for (int ch = 0; ch < BN / 64; ++ch) {
        const int f0 = T.n0 + 64 * ch;
        if (f0 >= p.F) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int fc = f0 + 32 * h;
          uint4 zg[4], zu[4];
          if (row_ok) {
            const uint4* pg = reinterpret_cast<const uint4*>(p.aux + r * 2 * p.F + fc);
            const uint4* pu = reinterpret_cast<const uint4*>(p.aux + r * 2 * p.F + p.F + fc);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              zg[i] = __ldg(pg + i);
              zu[i] = __ldg(pu + i);
            }
          }
          tmem_ld_32x32b_x32(tbase + 64 * ch + 32 * h, v);
          tmem_ld_wait();
          if (row_ok) {
            uint32_t wg[16], wu[16];
            swiglu_bwd32(v, zg, zu, wg, wu);
            store_row32(p.out0 + r * 2 * p.F + fc, wg);
            store_row32(p.out0 + r * 2 * p.F + p.F + fc, wu);
          }
        }
      }
    } else if constexpr (KIND == static_cast<int>(GemmKind::kDlhsFc2)) {
      const bool fused = p.aux != nullptr;
      for (int ch = 0; ch < BN / 64; ++ch) {
        const int f0 = T.n0 + 64 * ch;
        if (f0 >= p.F) break;
        uint8_t* gb = nullptr;
        if (full) gb = fused ? c.ring.template take<2>(lane) : c.ring.template take<1>(lane);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int fc = f0 + 32 * h;
          uint4 zg[4], zu[4];
          if (fused && row_ok) {
            const uint4* pg = reinterpret_cast<const uint4*>(p.aux + r * 2 * p.F + fc);
            const uint4* pu = reinterpret_cast<const uint4*>(p.aux + r * 2 * p.F + p.F + fc);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              zg[i] = __ldg(pg + i);
              zu[i] = __ldg(pu + i);
            }
          }
          tmem_ld_32x32b_x32(tbase + 64 * ch + 32 * h, v);
          tmem_ld_wait();
          if (fused) {
            uint32_t wg[16], wu[16];
            if (row_ok) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t gq[4] = {zg[i].x, zg[i].y, zg[i].z, zg[i].w};
                const uint32_t uq[4] = {zu[i].x, zu[i].y, zu[i].z, zu[i].w};
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                  float rg[2], ru[2];
#pragma unroll
                  for (int hh = 0; hh < 2; ++hh) {
                    const float dh = __uint_as_float(v[8 * i + 2 * qq + hh]);
                    const float g = hh ? bf16hi(gq[qq]) : bf16lo(gq[qq]);
                    const float u = hh ? bf16hi(uq[qq]) : bf16lo(uq[qq]);
                    const float sg = sigmoid_fast(g);
                    rg[hh] = dh * u * sg * (1.0f + g * (1.0f - sg));
                    ru[hh] = dh * g * sg;
                  }
                  wg[4 * i + qq] = pack_bf16x2(rg[0], rg[1]);
                  wu[4 * i + qq] = pack_bf16x2(ru[0], ru[1]);
                }
              }
            }
            if (full) {
              put_half(gb, lane, h, wg);
              put_half(c.ring.after(gb, 1), lane, h, wu);
            } else if (row_ok) {
              store_row32(p.out0 + r * 2 * p.F + fc, wg);
              store_row32(p.out0 + r * 2 * p.F + p.F + fc, wu);
            }
          } else {
            pack16(v, w);
            if (full) put_half(gb, lane, h, w);
            else if (row_ok) store_row32(p.out0 + r * p.F + fc, w);
          }
        }
        if (full) {
          publish();
          if (fused) flush_3d(gb, c.map_c, f0, y, 0, lane);  // dgate, dup
          else flush_2d(gb, c.map_c, f0, y, lane);
        }
      }
    } else if constexpr (KIND == static_cast<int>(GemmKind::kFc2Combine)) {
      // the combine, in place of a stored ys: each row's fp32 output times
      // its routing weight goes into its token's fp32 accumulator,
      // acc[t] += w[t,k] * ys[r] (16-byte vector reductions)
      const int j = row_ok ? __ldg(p.row_src + r) : -1;
      const float wk = j >= 0 ? __ldg(p.wts + j) : 0.0f;
      float* dst = j >= 0 ? p.acc + static_cast<long>(j / p.Ktop) * p.N : nullptr;
      for (int ch = 0; ch < BN / 64; ++ch) {
        const int col = T.n0 + 64 * ch;
        if (col >= p.N) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tmem_ld_32x32b_x32(tbase + 64 * ch + 32 * h, v);
          tmem_ld_wait();
          if (j >= 0) {
            float4* o = reinterpret_cast<float4*>(dst + col + 32 * h);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              atomicAdd(o + i, make_float4(wk * __uint_as_float(v[4 * i]),
                                           wk * __uint_as_float(v[4 * i + 1]),
                                           wk * __uint_as_float(v[4 * i + 2]),
                                           wk * __uint_as_float(v[4 * i + 3])));
          }
        }
      }
    } else {
      // plain bf16 store: FC2 and the dlhs of FC1 (N = D columns)
      for (int ch = 0; ch < BN / 64; ++ch) {
        const int col = T.n0 + 64 * ch;
        if (col >= p.N) break;
        uint8_t* buf = full ? c.ring.template take<1>(lane) : nullptr;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tmem_ld_32x32b_x32(tbase + 64 * ch + 32 * h, v);
          tmem_ld_wait();
          pack16(v, w);
          if (full) put_half(buf, lane, h, w);
          else if (row_ok) store_row32(p.out0 + r * p.N + col + 32 * h, w);
        }
        if (full) {
          publish();
          flush_2d(buf, c.map_c, col, y, lane);
        }
      }
    }
  }
}

// An empty group's weight-gradient tile is zero.
template <int BN, int RING>
__device__ __forceinline__ void zero_tile(const Tile& T, EpiCtx<RING>& c, const Params& p) {
  const int y = T.m0 + 32 * c.q;
  if (y >= p.M) return;
  for (int ch = 0; ch < BN / 64; ++ch) {
    const int col = T.n0 + 64 * ch;
    if (col >= p.N) break;
    uint8_t* buf = c.ring.template take<1>(c.lane);
    uint4* row = reinterpret_cast<uint4*>(buf + c.lane * 128);
#pragma unroll
    for (int j = 0; j < 8; ++j) row[j] = make_uint4(0u, 0u, 0u, 0u);
    publish();
    flush_3d(buf, c.map_c, col, y, T.e, c.lane);
  }
}

// ------------------------------------------------------------------ kernel
template <int KIND, class S>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_c,
                        const __grid_constant__ CUtensorMap map_d, const Params p) {
  constexpr int BN = S::BN;
  constexpr int CG = S::CG;
  constexpr int RING = S::kRing;
  using Tr = Traits<KIND, BN, CG>;
  constexpr int NACC = S::kNacc;
  constexpr int BNT = BN * NACC;  // tile width in output columns
  static_assert(NACC == 1 || Tr::kGroupedK, "wide tiles are for drhs");
  constexpr int kStages = S::kStages;
  constexpr int kStageBytes = S::kStageBytes;
  constexpr uint32_t kTmemCols = S::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* epi = ring + kStages * kStageBytes;  // staging of the epilogue warps
  uint8_t* zarea = epi + S::kEpiBytes;           // z rows of the fused SwiGLU backward
  typename S::Ctl& s = *reinterpret_cast<typename S::Ctl*>(zarea + S::kZBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (CG == 2) ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = (rank == 0);
  const int unit = blockIdx.x / CG;  // this CTA's (pair's) index in the schedule
  const int units = gridDim.x / CG;

  // ---------------------------------------------------------------- set-up
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_a);
    tma_prefetch_map(&map_b);
    tma_prefetch_map(&map_c);
    tma_prefetch_map(&map_d);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], kEpiWarps * CG);
    }
    for (int i = 0; i < kEpiWarps; ++i) {
      mbar_init(&s.zbar[i][0], 1);
      mbar_init(&s.zbar[i][1], 1);
    }
    for (int i = 0; i < kSched; ++i) {
      mbar_init(&s.sfull[i], 1);
      mbar_init(&s.sempty[i], sched_readers<CG>());
    }
    s.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(&s.tmem_base, kTmemCols);
    tmem_relinquish<CG>();
  }
  if (warp == 2) {
    // group offsets and the prefix of (128*CG)-row blocks per group (warp scan)
    constexpr int kRowsPerBlock = BM * CG;
    const int E = p.E;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int local = 0;
    for (int e = e0; e < e1; ++e) {
      const int a = __ldg(p.offs + e), b = __ldg(p.offs + e + 1);
      s.off[e] = a;
      local += (b - a + kRowsPerBlock - 1) / kRowsPerBlock;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e1; ++e) {
      s.mt[e] = run;
      run += (__ldg(p.offs + e + 1) - __ldg(p.offs + e) + kRowsPerBlock - 1) / kRowsPerBlock;
    }
    if (lane == 31) {
      s.mt[E] = incl;
      s.off[E] = __ldg(p.offs + E);
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers exist before any remote arrive
  tc_fence_after();
  if constexpr (Tr::kGroupedK) sort_groups_desc(s, p.E);
  const uint32_t tmem_base = s.tmem_base;
  const WaitCtl wc{&s.abort_flag, p.status, p.limit_ns};
  const int ntiles = total_tiles<KIND, BNT, CG>(p, s);
  // drhs tiles come from the dynamic schedule, the others in a fixed stride
  constexpr bool kDyn = Tr::kGroupedK;
  uint32_t sseq = 0;      // dynamic: slots read (or written) so far
  int tstat = unit;       // fixed: this unit's next tile

  if (warp == 0 && KIND == static_cast<int>(GemmKind::kFc1Gather)) {
    // ----------------------------------------- producer (gathered FC1 rows)
    // The whole warp: lane 0 waits for a free stage, arms it with the whole
    // stage's bytes and loads the B operand; then lane i gathers A rows
    // 4i..4i+3 of the tile straight from the token-major x (row r of the
    // tile is token row_src[r] / K) with one TMA gather of four 128-byte
    // rows, which lands in the 128-byte-swizzled layout the MMA reads.
    if constexpr (KIND == static_cast<int>(GemmKind::kFc1Gather) && CG == 1) {
      uint32_t stage = 0, phase = 0, nfill = 0;  // stages filled so far
      bool aborted = false;
      while (!aborted) {
        const int t = tstat;
        tstat += units;
        if (t >= ntiles) break;
        const Tile T = decode_tile<KIND, BNT, CG>(t, rank, p, s);
        // this lane's four rows (rows past the last are gathered from token
        // 0 and never stored)
        int tok[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const long r = static_cast<long>(T.row0) + 4 * lane + q;
          tok[q] = 0;
          if (r < p.R) {
            const int j = __ldg(p.row_src + r);
            tok[q] = j >= 0 ? j / p.Ktop : 0;
          }
        }
        const uint32_t tx_bytes = stage_bytes<KIND, BN, CG, NACC>(T, p);
        for (int kb = 0; kb < T.kb; ++kb) {
          bool ok = true;
          if (lane == 0) ok = mbar_wait(&s.empty[stage], phase ^ 1u, wc);
          if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { aborted = true; break; }
          uint8_t* sa = ring + stage * kStageBytes;
          if (lane == 0) {
            mbar_arrive_expect_tx(&s.full[stage], tx_bytes);
            issue_loads<KIND, BN, CG, NACC>(T, kb, rank, sa, sa + kAStageBytes,
                                            smem_u32(&s.full[stage]), &map_a, &map_b, &map_d, p);
          }
          ++nfill;
          __syncwarp();  // the stage is armed before any gather lands
          tma_gather4(sa + 512 * lane, &map_a, smem_u32(&s.full[stage]), kb * BK, tok[0], tok[1],
                      tok[2], tok[3]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (aborted && lane == 0) {  // the copies of stages in flight land before the CTA exits
        for (uint32_t i = 0; i < kStages; ++i) {
          const uint32_t f = ring_uses(nfill, i, kStages);
          if (f > 0) (void)mbar_wait_drain(&s.full[i], (f - 1u) & 1u, 100000000ull);
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // For a pair, both CTAs' bytes complete on the even CTA's full barrier,
      // which the even CTA arms with the bytes of both.
      uint32_t stage = 0, phase = 0, nfill = 0;  // stages filled so far
      const uint32_t full0 = (CG == 2) ? mapa_shared(smem_u32(&s.full[0]), 0) : smem_u32(&s.full[0]);
      bool aborted = false;
      // dynamic schedule: the even CTA claims the next tile a little before
      // the current one's loads end (the atomic's latency hides behind them)
      int claimed = (kDyn && leader) ? static_cast<int>(atomicAdd(p.tile_ctr, 1u)) : 0;
      while (!aborted) {
        int t;
        if constexpr (!kDyn) {
          t = tstat;
          tstat += units;
        } else if (leader) {
          t = claimed;
          if (!sched_publish<CG>(s, sseq, t, wc)) { aborted = true; break; }
        } else {
          t = sched_take<CG>(s, sseq, leader, true, 1u, wc);
          if (t < 0) { aborted = true; break; }
        }
        if (t >= ntiles) break;
        const Tile T = decode_tile<KIND, BNT, CG>(t, rank, p, s);
        const uint32_t tx_bytes = stage_bytes<KIND, BN, CG, NACC>(T, p) * CG;
        bool next_claimed = !(kDyn && leader);
        for (int kb = 0; kb < T.kb; ++kb) {
          if (!next_claimed && kb + 2 >= T.kb) {
            claimed = static_cast<int>(atomicAdd(p.tile_ctr, 1u));
            next_claimed = true;
          }
          if (!mbar_wait(&s.empty[stage], phase ^ 1u, wc)) { aborted = true; break; }
          uint8_t* sa = ring + stage * kStageBytes;
          if (leader) mbar_arrive_expect_tx(&s.full[stage], tx_bytes);
          issue_loads<KIND, BN, CG, NACC>(T, kb, rank, sa, sa + kAStageBytes,
                                          full0 + stage * static_cast<uint32_t>(sizeof(uint64_t)),
                                          &map_a, &map_b, &map_d, p);
          ++nfill;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!next_claimed) claimed = static_cast<int>(atomicAdd(p.tile_ctr, 1u));
      }
      if (aborted && leader) {  // let copies already in flight land before the CTA exits
        for (uint32_t i = 0; i < kStages; ++i) {
          const uint32_t f = ring_uses(nfill, i, kStages);
          if (f > 0) (void)mbar_wait_drain(&s.full[i], (f - 1u) & 1u, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (CG == 1 || leader) {
      // ----------------------------------------------------------- MMA
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      uint32_t ncommit = 0;  // stages whose MMAs were committed so far
      bool aborted = false;
      while (!aborted) {
        int t;
        if constexpr (!kDyn) {
          t = tstat;
          tstat += units;
        } else {
          t = sched_take<CG>(s, sseq, leader, lane == 0, 0xffffffffu, wc);
          if (t < 0) { aborted = true; break; }
        }
        if (t >= ntiles) break;
        const Tile T = decode_tile<KIND, BNT, CG>(t, rank, p, s);
        if (T.kb == 0) continue;
        if (!__all_sync(0xffffffffu, mbar_wait(&s.tempty[acc], acc_phase ^ 1u, wc))) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * S::kAccStride;
        // a lone CTA's narrow FC1 tile reads the first gate and the first up
        // chunk, which the boxes left two chunks apart
        const uint32_t b_lbo = (fc1_like<KIND>() && CG == 1 &&
                                acc_cols<KIND, BN, CG>(T, 0, p) < BN)
                                   ? 2 * kChunkBytes
                                   : kChunkBytes;
        uint32_t idesc[NACC];  // instruction descriptors with each accumulator's MMA width
#pragma unroll
        for (int a = 0; a < NACC; ++a)
          idesc[a] = (Tr::kIdesc & ~(0x3Fu << 17)) |
                     (static_cast<uint32_t>(acc_cols<KIND, BN, CG>(T, a, p) >> 3) << 17);
        for (int kb = 0; kb < T.kb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&s.full[stage], phase, wc))) {
            aborted = true;
            break;
          }
          tc_fence_after();
          uint8_t* sa = ring + stage * kStageBytes;
          uint8_t* sb = sa + kAStageBytes;
          int ksteps = BK / kUmmaK;
          if constexpr (Tr::kGroupedK) {
            const int valid = T.klen - kb * BK;
            if (valid < BK) {
              zero_tail<BN, CG, NACC>(sa, sb, valid, lane);
              ksteps = (valid + kUmmaK - 1) / kUmmaK;
            }
          }
          __syncwarp();
          if (lane == 0) {
            const uint32_t a_addr = smem_u32(sa);
            const uint32_t b_addr = smem_u32(sb);
#pragma unroll
            for (int kk = 0; kk < BK / kUmmaK; ++kk) {
              if (kk >= ksteps) break;
              const uint64_t ad = Tr::kAMn
                                      ? smem_desc_sw128(a_addr + kk * 2048, kChunkBytes, 1024)
                                      : smem_desc_sw128(a_addr + kk * 32, 16, 1024);
#pragma unroll
              for (int a = 0; a < NACC; ++a) {
                if (a > 0 && (idesc[a] & (0x3Fu << 17)) == 0) break;  // nothing valid
                const uint32_t b_acc = b_addr + a * (BN / CG) * BK * 2;
                const uint64_t bd = Tr::kBMn ? smem_desc_sw128(b_acc + kk * 2048, b_lbo, 1024)
                                             : smem_desc_sw128(b_acc + kk * 32, 16, 1024);
                umma_bf16<CG>(d_tmem + a * BN, ad, bd, idesc[a], (kb > 0 || kk > 0) ? 1u : 0u);
              }
            }
            umma_commit<CG>(&s.empty[stage]);
          }
          __syncwarp();
          ++ncommit;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (aborted) break;
        if (lane == 0) umma_commit<CG>(&s.tfull[acc]);
        __syncwarp();
        if (++acc == S::kAccSlots) { acc = 0; acc_phase ^= 1u; }
      }
      if (aborted && ncommit > 0) {  // let issued MMAs finish before TMEM is freed
        const uint32_t last = (ncommit - 1u) % kStages;
        (void)mbar_wait_drain(&s.empty[last], (ring_uses(ncommit, last, kStages) - 1u) & 1u,
                              100000000ull);
      }
    }
    // the odd CTA's MMA warp only takes part in the collective TMEM allocation
  } else {
    // -------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    EpiCtx<RING> ec{&map_c, &map_d, Ring<RING>{epi + (warp - 2) * RING * kBufBytes, 0u}, q, lane,
                    ZPipe{zarea + (warp - 2) * S::kZSlots * 2 * S::kZBuf, &s.zbar[warp - 2][0],
                          0u, 0, 0, 0, -1, 0},
                    &wc};
    uint32_t tempty_peer = 0;
    if constexpr (CG == 2) tempty_peer = mapa_shared(smem_u32(&s.tempty[0]), 0);
    uint32_t acc = 0, acc_phase = 0;
    for (;;) {
      int t;
      if constexpr (!kDyn) {
        t = tstat;
        tstat += units;
      } else {
        t = sched_take<CG>(s, sseq, leader, lane == 0, 0xffffffffu, wc);
        if (t < 0) break;
      }
      if (t >= ntiles) break;
      const Tile T = decode_tile<KIND, BNT, CG>(t, rank, p, s);
      if (T.kb == 0) {
        if constexpr (Tr::kGroupedK) {
#pragma unroll
          for (int a = 0; a < NACC; ++a) {
            Tile Ta = T;
            Ta.n0 = T.n0 + a * BN;
            zero_tile<BN, RING>(Ta, ec, p);
          }
        }
        continue;
      }
      // the fused SwiGLU backward's z: the tile's first chunks are requested
      // before its accumulator is waited for (if the previous tile has not
      // requested them already), with the warp's next tile known
      int tn = -1;
      Tile Tn{};
      if constexpr (S::kZB) {
        if (z_by_tma<KIND, true, RING>(T, ec, p)) {
          if (tstat < ntiles) {
            tn = tstat;
            Tn = decode_tile<KIND, BNT, CG>(tn, rank, p, s);
          }
          if (ec.zp.qt != t) {
            ec.zp.qt = t;
            ec.zp.qch = 0;
          }
          z_fill<KIND, BN, true, RING, S::kZW>(t, T, tn, Tn, ec, p);
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&s.tfull[acc], acc_phase, wc))) break;
      tc_fence_after();
#pragma unroll
      for (int a = 0; a < NACC; ++a) {
        Tile Ta = T;
        Ta.n0 = T.n0 + a * BN;
        epilogue_tile<KIND, BN, CG, RING, S::kZB, S::kZW>(
            Ta, tmem_base + acc * S::kAccStride + a * BN + (static_cast<uint32_t>(q * 32) << 16),
            ec, p, t, tn, Tn);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CG == 2 && !leader)
          mbar_arrive_remote(tempty_peer + acc * static_cast<uint32_t>(sizeof(uint64_t)));
        else
          mbar_arrive(&s.tempty[acc]);
      }
      if (++acc == S::kAccSlots) { acc = 0; acc_phase ^= 1u; }
    }
    z_drain(ec);                     // z requests still in flight land (abort)
    if (lane == 0) bulk_wait_all();  // every store has finished before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // both CTAs are done with each other's memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, kTmemCols);
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

// bf16 tensor map, dims innermost first; strides in bytes for dims 1..rank-1.
// The swizzle span must equal the box's inner extent in bytes (128 or 64).
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t gd[4], gs[3];
  cuuint32_t bd[4], es[4] = {1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bd[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gd, gs, bd, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
           uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {inner * 2};
  const uint32_t box[2] = {box_inner, box_outer};
  return make_map(m, base, 2, dims, strides, box);
}

bool map3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
           uint32_t box_inner, uint32_t box_mid) {
  const uint64_t dims[3] = {inner, mid, outer};
  const uint64_t strides[2] = {inner * 2, inner * mid * 2};
  const uint32_t box[3] = {box_inner, box_mid, 1};
  return make_map(m, base, 3, dims, strides, box);
}

// A [rows][2F] tensor of gate and up halves (z, dz) seen as [2][rows][F]:
// one box of 32 rows x `cols` columns per half moves a gate chunk and the up
// chunk F columns to its right with one instruction, into two consecutive
// staging buffers (4 KB with 128-byte rows at 64 columns, 2 KB with 64-byte
// rows at 32).  Dims (innermost first): F, rows, 2.
bool map_halves(CUtensorMap* m, const void* base, uint64_t F, uint64_t rows, uint32_t cols = 64) {
  const uint64_t dims[3] = {F, rows, 2};
  const uint64_t strides[2] = {4 * F, 2 * F};
  const uint32_t box[3] = {cols, 32, 2};
  return make_map(m, base, 3, dims, strides, box,
                  cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// An MN-major operand [outer][rows][inner] (inner contiguous, a multiple of
// 64) seen as [outer][inner/64][rows][64]: one box of `box_chunks` 64-wide
// chunks x 64 rows lands as consecutive 8 KB chunks, the layout the MMA
// descriptors expect.  Dims (innermost first): 64, rows, chunks[, outer].
// The map's rank must match the load instruction: 4 for the per-expert
// weights (loaded with 4-D coordinates even when E = 1), 3 for a 2-D operand.
bool map_chunks(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t outer,
                uint32_t box_chunks, int rank) {
  const uint64_t dims[4] = {64, rows, inner / 64, outer};
  const uint64_t strides[3] = {inner * 2, 128, inner * rows * 2};
  const uint32_t box[4] = {64, 64, box_chunks, 1};
  return make_map(m, base, rank, dims, strides, box);
}

template <int KIND, class S>
cudaError_t launch_kind(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                        const CUtensorMap& md, const Params& p, long max_units, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<KIND, S>;
  constexpr size_t bytes = S::kSmemBytes;
  // the shared-memory opt-in is set once per device (not on every launch, so
  // that launches being captured into a CUDA graph make no such call)
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err != cudaSuccess) return err;
    attr_set[dev].store(true, std::memory_order_release);
  }
  long units = sm_count() / S::CG;
  if (max_units < units) units = max_units;
  if (units <= 0) return cudaSuccess;
  if constexpr (S::CG == 1) {
    kern<<<static_cast<int>(units), kThreads, bytes, s>>>(ma, mb, mc, md, p);
    return cudaGetLastError();
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // clusters that can be resident at once (one CTA per SM), cached per kernel
    static int max_clusters = 0;
    static std::once_flag once;
    std::call_once(once, [&] {
      cfg.gridDim = dim3(static_cast<unsigned>(2 * (sm_count() / 2)), 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) max_clusters = n;
      else max_clusters = sm_count() / 2;
    });
    if (units > max_clusters) units = max_clusters;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * units), 1, 1);
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, md, p);
  }
}

inline long cdiv(long a, long b) { return (a + b - 1) / b; }

// Operand/output maps and tile counts of one grouped GEMM, for CG CTAs per MMA.
template <class S>
cudaError_t launch_shape(const GemmCall& c, cudaStream_t s) {
  constexpr int BN = S::BN;
  constexpr int CG = S::CG;
  constexpr uint32_t kBRows = BN / CG;
  const moe_dims& d = c.d;
  if (d.E > S::kMaxE) return cudaErrorInvalidValue;  // the control block's expert arrays
  const long R = static_cast<long>(d.T) * d.K;
  Params p{};
  // lone CTAs and groups of at most one 128-row block on average: each
  // expert's weights are read once
  p.evict_weights = (CG == 1 && R <= static_cast<long>(d.E) * BM) ? 1 : 0;
  p.offs = c.offs;
  p.out0 = static_cast<__nv_bfloat16*>(c.out0);
  p.out1 = static_cast<__nv_bfloat16*>(c.out1);
  p.aux = static_cast<const __nv_bfloat16*>(c.aux);
  p.status = c.dev_status;
  p.tile_ctr = c.tile_ctr;
  p.limit_ns = kDefaultWaitLimitNs;
  p.E = d.E;
  p.F = d.F;
  CUtensorMap ma, mb, mc, md;
  bool ok = false;
  const long row_blocks_bound = R / (BM * CG) + d.E;
  const long F2 = 2L * d.F;
  if constexpr (S::kZB) {
    // shapes with z slots run only the FC2 dlhs with the fused SwiGLU backward
    if (c.kind != GemmKind::kDlhsFc2 || c.aux == nullptr) return cudaErrorInvalidValue;
    p.Kdim = d.D;
    p.N = d.F;
    p.n_tiles = static_cast<int>(cdiv(d.F, BN));
    ok = map2d(&ma, c.a, d.D, R, 64, BM) && map3d(&mb, c.b, d.D, d.F, d.E, 64, kBRows) &&
         map_halves(&mc, c.out0, d.F, R, S::kZW) && map_halves(&md, c.aux, d.F, R, S::kZW);
    if (!ok) return cudaErrorInvalidValue;
    return launch_kind<2, S>(ma, mb, mc, md, p, row_blocks_bound * p.n_tiles, s);
  } else {
    switch (c.kind) {
      case GemmKind::kFc1:
      case GemmKind::kFc2:
      case GemmKind::kDlhsFc2:
      case GemmKind::kDlhsFc1:
      case GemmKind::kFc1Gather:
      case GemmKind::kFc2Combine:
        if constexpr (S::kNacc == 1) {
          switch (c.kind) {
            case GemmKind::kFc1:
              // h, z gate and z up are staged together, z gate and z up in
              // adjacent buffers (one 3-D store): the ring holds whole triples
              if constexpr (S::kRing % 3 == 0) {
                p.Kdim = d.D;
                p.N = d.F;
                p.n_tiles = static_cast<int>(cdiv(d.F, BN / 2));
                ok = map2d(&ma, c.a, d.D, R, 64, BM) &&
                     map_chunks(&mb, c.b, F2, d.D, d.E, BN / 64 / 2, 4) &&
                     map2d(&mc, c.out0, d.F, R, 64, 32);
                if (ok) ok = (c.out1 != nullptr) ? map_halves(&md, c.out1, d.F, R) : (md = mc, true);
                if (!ok) return cudaErrorInvalidValue;
                return launch_kind<0, S>(ma, mb, mc, md, p, row_blocks_bound * p.n_tiles, s);
              }
              return cudaErrorInvalidValue;
            case GemmKind::kFc2:
              p.Kdim = d.F;
              p.N = d.D;
              p.n_tiles = static_cast<int>(cdiv(d.D, BN));
              ok = map2d(&ma, c.a, d.F, R, 64, BM) &&
                   map_chunks(&mb, c.b, d.D, d.F, d.E, BN / 64 / CG, 4) &&
                   map2d(&mc, c.out0, d.D, R, 64, 32) && map3d(&md, c.b, d.D, d.F, d.E, 64, 64);
              if (!ok) return cudaErrorInvalidValue;
              return launch_kind<1, S>(ma, mb, mc, md, p, row_blocks_bound * p.n_tiles, s);
            case GemmKind::kDlhsFc2:
              // fused, dgate and dup are staged together in adjacent buffers
              // (one 3-D store): the ring must hold whole pairs
              if (c.aux != nullptr && S::kRing % 2 != 0) return cudaErrorInvalidValue;
              if constexpr (S::kRing >= 2) {
                p.Kdim = d.D;
                p.N = d.F;
                p.n_tiles = static_cast<int>(cdiv(d.F, BN));
                ok = map2d(&ma, c.a, d.D, R, 64, BM) && map3d(&mb, c.b, d.D, d.F, d.E, 64, kBRows) &&
                     (c.aux != nullptr ? map_halves(&mc, c.out0, d.F, R)
                                       : map2d(&mc, c.out0, d.F, R, 64, 32));
                if (ok) ok = (c.aux != nullptr) ? map_halves(&md, c.aux, d.F, R) : (md = mc, true);
                if (!ok) return cudaErrorInvalidValue;
                return launch_kind<2, S>(ma, mb, mc, md, p, row_blocks_bound * p.n_tiles, s);
              }
              return cudaErrorInvalidValue;
            case GemmKind::kDlhsFc1:
              p.Kdim = 2 * d.F;
              p.N = d.D;
              p.n_tiles = static_cast<int>(cdiv(d.D, BN));
              ok = map2d(&ma, c.a, F2, R, 64, BM) && map3d(&mb, c.b, F2, d.D, d.E, 64, kBRows) &&
                   map2d(&mc, c.out0, d.D, R, 64, 32);
              if (!ok) return cudaErrorInvalidValue;
              return launch_kind<3, S>(ma, mb, mc, mc, p, row_blocks_bound * p.n_tiles, s);
            case GemmKind::kFc1Gather:
              // FC1 on rows gathered from x by row_src (single CTAs); the A
              // map is x [T][D] with a box of one row, for four-row gathers
              if constexpr (S::CG == 1 && S::kRing % 3 == 0) {
                p.Kdim = d.D;
                p.N = d.F;
                p.n_tiles = static_cast<int>(cdiv(d.F, BN / 2));
                p.row_src = c.row_src;
                p.Ktop = d.K;
                p.R = R;
                ok = map2d(&ma, c.a, d.D, d.T, 64, 1) &&
                     map_chunks(&mb, c.b, F2, d.D, d.E, BN / 64 / 2, 4) &&
                     map2d(&mc, c.out0, d.F, R, 64, 32);
                if (ok) ok = (c.out1 != nullptr) ? map_halves(&md, c.out1, d.F, R) : (md = mc, true);
                if (!ok || c.row_src == nullptr) return cudaErrorInvalidValue;
                return launch_kind<6, S>(ma, mb, mc, md, p, row_blocks_bound * p.n_tiles, s);
              }
              return cudaErrorInvalidValue;
            case GemmKind::kFc2Combine:
              // FC2 whose rows go, weighted, into the fp32 accumulator
              // (single CTAs); no output map
              if constexpr (S::CG == 1) {
                p.Kdim = d.F;
                p.N = d.D;
                p.n_tiles = static_cast<int>(cdiv(d.D, BN));
                p.row_src = c.row_src;
                p.wts = c.w;
                p.acc = c.acc;
                p.Ktop = d.K;
                p.R = R;
                ok = map2d(&ma, c.a, d.F, R, 64, BM) &&
                     map_chunks(&mb, c.b, d.D, d.F, d.E, BN / 64 / CG, 4) &&
                     map3d(&md, c.b, d.D, d.F, d.E, 64, 64);
                if (!ok || c.row_src == nullptr || c.w == nullptr || c.acc == nullptr)
                  return cudaErrorInvalidValue;
                return launch_kind<7, S>(ma, mb, ma, md, p, row_blocks_bound * p.n_tiles, s);
              }
              return cudaErrorInvalidValue;
            default:
              break;
          }
        }
        return cudaErrorInvalidValue;
      case GemmKind::kDrhsFc2:
        p.M = d.F;
        p.N = d.D;
        p.m_tiles = static_cast<int>(cdiv(d.F, BM * CG));
        p.n_tiles = static_cast<int>(cdiv(d.D, BN * S::kNacc));
        ok = map_chunks(&ma, c.a, d.F, R, 1, 2, 3) && map_chunks(&mb, c.b, d.D, R, 1, BN / 64 / CG, 3) &&
             map3d(&mc, c.out0, d.D, d.F, d.E, 64, 32) && map2d(&md, c.b, d.D, R, 64, 64);
        if (!ok || c.tile_ctr == nullptr) return cudaErrorInvalidValue;
        if (cudaError_t e = cudaMemsetAsync(c.tile_ctr, 0, sizeof(unsigned int), s); e != cudaSuccess)
          return e;
        return launch_kind<4, S>(ma, mb, mc, md, p, static_cast<long>(d.E) * p.m_tiles * p.n_tiles,
                                 s);
      case GemmKind::kDrhsFc1:
        p.M = d.D;
        p.N = 2 * d.F;
        p.m_tiles = static_cast<int>(cdiv(d.D, BM * CG));
        p.n_tiles = static_cast<int>(cdiv(F2, BN * S::kNacc));
        ok = map_chunks(&ma, c.a, d.D, R, 1, 2, 3) && map_chunks(&mb, c.b, F2, R, 1, BN / 64 / CG, 3) &&
             map3d(&mc, c.out0, F2, d.D, d.E, 64, 32) && map2d(&md, c.b, F2, R, 64, 64);
        if (!ok || c.tile_ctr == nullptr) return cudaErrorInvalidValue;
        if (cudaError_t e = cudaMemsetAsync(c.tile_ctr, 0, sizeof(unsigned int), s); e != cudaSuccess)
          return e;
        return launch_kind<5, S>(ma, mb, mc, md, p, static_cast<long>(d.E) * p.m_tiles * p.n_tiles,
                                 s);
    }
  }
  return cudaErrorInvalidValue;
}

// Single-CTA shape: 3 stages of 48 KB and 3 staging buffers per warp.
using Shape1 = Shape<256, 3, 1, 3>;
// Lone-CTA drhs: a fourth operand stage in place of two of each epilogue
// warp's staging buffers.  Short groups make these tiles a few k-blocks
// long, each loading 48 KB of operands for 512 MMA cycles, and the feed is
// bound by the bytes in flight: at E=256 experts of ~256 rows, FC1 drhs
// 4.72 -> 4.07-4.25 ms, FC2 drhs 2.30 -> 1.94-2.13 ms.  (Two CTAs of a
// cluster sharing B by TMA multicast were slower, 5.12 ms, as were CTA
// pairs, 5.07 ms: both tie each stage to the slower of two CTAs.)
using Shape1Drhs = Shape<256, 4, 1, 1>;
// CTA-pair shapes: stages of 32 KB per CTA.  FC1 stages three buffers at once
// (h, z gate, z up); the others need at most two.  FC1's fifth stage (paid
// for with its fourth staging buffer) cuts the MMA's waits for operands from
// 20% to 16% of the kernel and its cycles by 5%.
using Shape2Fc1 = Shape<256, 5, 2, 3>;
using Shape2 = Shape<256, 5, 2, 2>;
// With the control block's expert arrays for at most 128 experts a sixth
// stage fits (E=128, ~2048 rows per expert: FC2 688 -> 674 us, FC2 drhs as
// 256-wide pairs 687 -> 664 us, FC1 dlhs unchanged).
using Shape2E128 = Shape<256, 6, 2, 2, 0, 1, 128>;
// drhs: tiles two accumulators wide (fewer bytes loaded per MMA).
using Shape2Drhs = Shape<256, 3, 2, 2, 0, 2>;
// ... and a fourth stage for at most 128 experts (FC1 drhs 1243 -> 1219 us).
using Shape2DrhsE128 = Shape<256, 4, 2, 2, 0, 2, 128>;
// The FC2 dlhs with the fused SwiGLU backward: two z slots per epilogue
// warp, in which dz is also staged (no staging ring).  Its operand feed is
// bound by the bytes in flight up to five stages (E=128, ~2048 rows per
// expert: 966 us with three stages, 845 with four, 791 with five; a sixth
// measured the same, 806 vs 807-813 us), so the slots hold 32-column chunks
// (32 KB for the four warps instead of 64) and the space goes to the operand
// ring: six stages on pairs when the control block's expert arrays hold at
// most 128 experts, five (instead of four) for up to 1024 (E=256, ~256 rows
// per expert: 2095-2111 -> 1885-1890 us, same box); a lone CTA's 48 KB
// stages fit four times with 128 experts, three times (beside 64-column
// slots) with 1024.
using Shape1Dz = Shape<256, 3, 1, 0, 2>;
using Shape1DzE128 = Shape<256, 4, 1, 0, 2, 1, 128, 32>;
using Shape2Dz = Shape<256, 5, 2, 0, 2, 1, kMaxExperts, 32>;
using Shape2DzE128 = Shape<256, 6, 2, 0, 2, 1, 128, 32>;

// Whether a grouped GEMM runs on CTA pairs.  The pair's 256-row block is the
// unit of rows for the forward and dlhs GEMMs; pairs pay off from ~256 rows
// per group (2048 tokens, E=128, top-8: 128 rows, FC1 167 us alone, 176 us
// on pairs; 4096 tokens: 226 vs 223 us; 8192 tokens: 352 vs 333 us).  drhs
// tiles reduce over their group's rows: with short groups (a few 64-row
// blocks per tile) a tile is mostly epilogue, and single CTAs with
// double-buffered accumulators do best (E=256 experts of ~256 rows: FC1
// drhs 4.1-4.3 ms alone, 5.1 ms as 256-wide pairs, 5.6 ms as 512-wide pairs);
// from ~1024 rows per group 512-wide pair tiles do (E=128 of ~2048 rows:
// the step takes 7.73 ms with them, 8.07 ms with 256-wide pair tiles).
// MOE_GEMM_PAIR=0/1 forces the choice.
bool use_pairs(const GemmCall& c) {
  const char* env = std::getenv("MOE_GEMM_PAIR");
  if (env != nullptr && env[0] == '0') return false;
  if (env != nullptr && env[0] == '1') return true;
  const long rows_per_group = static_cast<long>(c.d.T) * c.d.K / c.d.E;
  const bool drhs = c.kind == GemmKind::kDrhsFc2 || c.kind == GemmKind::kDrhsFc1;
  return rows_per_group >= (drhs ? 1024 : 256);
}

// Whether drhs tiles on pairs are 512 columns wide (two accumulators, one
// TMEM slot) rather than 256 (double-buffered).  MOE_GEMM_WIDE=0/1 forces it.
bool wide_drhs(const GemmCall& c) {
  const char* env = std::getenv("MOE_GEMM_WIDE");
  if (env != nullptr && env[0] == '0') return false;
  if (env != nullptr && env[0] == '1') return true;
  (void)c;
  return true;
}

}  // namespace

cudaError_t launch_grouped_gemm(const GemmCall& c, cudaStream_t s) {
  const moe_dims& d = c.d;
  const long R = static_cast<long>(d.T) * d.K;
  if (R == 0) {
    // no rows: forward/dlhs outputs are empty; weight gradients are zero
    if (c.kind == GemmKind::kDrhsFc2)
      return cudaMemsetAsync(c.out0, 0, static_cast<size_t>(d.E) * d.F * d.D * 2, s);
    if (c.kind == GemmKind::kDrhsFc1)
      return cudaMemsetAsync(c.out0, 0, static_cast<size_t>(d.E) * d.D * 2 * d.F * 2, s);
    return cudaSuccess;
  }
  // the gathered FC1 and the combined FC2 run on single CTAs (their A rows
  // and output rows are per token, not per pair of CTAs)
  if (c.kind == GemmKind::kFc1Gather || c.kind == GemmKind::kFc2Combine)
    return launch_shape<Shape1>(c, s);
  const bool dz = (c.kind == GemmKind::kDlhsFc2 && c.aux != nullptr);
  const bool drhs = c.kind == GemmKind::kDrhsFc2 || c.kind == GemmKind::kDrhsFc1;
  const bool e128 = d.E <= 128;  // the shapes whose control block holds 128 experts
  if (!use_pairs(c)) {
    if (drhs) return launch_shape<Shape1Drhs>(c, s);
    if (dz) return e128 ? launch_shape<Shape1DzE128>(c, s) : launch_shape<Shape1Dz>(c, s);
    return launch_shape<Shape1>(c, s);
  }
  if (drhs) {
    if (wide_drhs(c)) return e128 ? launch_shape<Shape2DrhsE128>(c, s) : launch_shape<Shape2Drhs>(c, s);
    return e128 ? launch_shape<Shape2E128>(c, s) : launch_shape<Shape2>(c, s);
  }
  if (c.kind == GemmKind::kFc1) return launch_shape<Shape2Fc1>(c, s);
  if (dz) return e128 ? launch_shape<Shape2DzE128>(c, s) : launch_shape<Shape2Dz>(c, s);
  return e128 ? launch_shape<Shape2E128>(c, s) : launch_shape<Shape2>(c, s);
}

}  // namespace moe
