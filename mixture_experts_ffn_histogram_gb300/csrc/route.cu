// Routing and group_size histogram of the MoE block.
//
// MaxText "Gemma4 26B MoE on TPU v6e: MaxText layer/model optimizations",
// Commits table row 6: top_k_weights and group_size are computed next to the
// rest of the block; MaxText "MoE: fused TensorCore Pallas permute/combine
// kernels and split-expert wi layout for TPU v6e", Commits table row 2: the
// group_size histogram is computed before the token gather.
//
// One kernel, three phases; deterministic (no atomic decides an order):
//   1. Each warp owns a contiguous run of tokens.  For each of them a group
//      of G lanes selects the top-K scores by K rounds of a group-wide
//      (score desc, id asc) arg-max and computes the routing weights (or, for
//      given routing, reads the ids).  Each slot's rank among the warp's
//      earlier slots of the same expert (__match_any_sync over 32 slots at a
//      time, plus the warp's running count per expert in shared memory) is
//      stored in pos for now.  The block then turns the per-warp counts into
//      prefixes over its warps and publishes its per-expert totals.
//   2. After a barrier every block sums the published totals of the blocks
//      before it (its prefix per expert) and of all blocks (group_sizes),
//      and scans group_sizes over experts (group_offsets).
//   3. pos = group_offsets[e] + block prefix + warp prefix + rank in warp,
//      i.e. the stable order in the flat slot index t*K+k; row_src[pos] = j.
// Two forms of the barrier and the exchange of totals: with few tokens the
// grid is one thread-block cluster (hardware cluster barrier, totals read
// from the other blocks' shared memory); otherwise a cooperative launch
// (every block resident at once; a grid barrier on one word of global
// scratch, totals through global memory).  Either kernel is the call's only
// launch, and both give the same outputs bit for bit.
#include <cuda.h>

#include <atomic>
#include <cfloat>
#include <climits>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRouteMaxWarps = 16;

// The two halves of a cluster barrier, for work between them: arrive
// orders this thread's earlier accesses before the others' wait returns.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A score and its expert id as one 64-bit key whose unsigned order is the
// selection order (score descending, then id ascending): the score's bits
// made monotone (sign flipped for positives, all bits for negatives; -0 is
// first turned into +0 so that equal scores tie), and the id inverted in the
// low half.  Key 0 lies below every real key and stands for "no expert".
__device__ __forceinline__ uint64_t score_key(float v, int e) {
  uint32_t u = __float_as_uint(v + 0.0f);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(e));
}
__device__ __forceinline__ float key_score(uint64_t k) {
  const uint32_t u = static_cast<uint32_t>(k >> 32);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
__device__ __forceinline__ int key_expert(uint64_t k) {
  return static_cast<int>(~static_cast<uint32_t>(k));
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a cooperative launch on one 64-bit word: a tag
// (high half) and an arrival count (low half).  Every launch leaves the word
// at (tag, 0) for the next: the last block through clears the count.  A word
// that does not carry the tag (memory never used for this, or other data) is
// claimed by compare-and-swap, so it needs no clearing before the first use.
// Every block then waits (bounded) until the count reaches the number of
// blocks.  Returns false, after recording MOE_ERR_TIMEOUT, when a wait gave
// up; the word is then left in an unknown state.
constexpr uint32_t kBarrierTag = 0x5EC0DEu;

__device__ __forceinline__ bool grid_barrier(unsigned long long* word, uint32_t nblocks,
                                             int32_t* status, uint64_t limit_ns) {
  __shared__ int ok_flag;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned long long tagged = static_cast<unsigned long long>(kBarrierTag) << 32;
    bool ok = true;
    unsigned long long cur = atomicAdd(word, 1ull);
    if (static_cast<uint32_t>(cur >> 32) != kBarrierTag) {
      // the add landed on an untagged word: count this block into a tagged one
      ok = false;
      cur += 1ull;
      for (uint32_t it = 0; it < kMaxWaitIters; ++it) {
        const unsigned long long want =
            (static_cast<uint32_t>(cur >> 32) == kBarrierTag) ? cur + 1ull : tagged + 1ull;
        const unsigned long long got = atomicCAS(word, cur, want);
        if (got == cur) { ok = true; break; }
        cur = got;
      }
    }
    if (ok) {
      ok = false;
      const uint64_t start = global_timer_ns();
      for (uint32_t it = 0; it < kMaxWaitIters; ++it) {
        const unsigned long long v = ld_acquire_gpu_u64(word);
        if (static_cast<uint32_t>(v >> 32) == kBarrierTag && static_cast<uint32_t>(v) >= nblocks) {
          ok = true;
          break;
        }
        if ((it & 63u) == 63u && global_timer_ns() - start > limit_ns) break;
        __nanosleep(32);
      }
    }
    if (ok) {
      // leave: the last of the blocks to leave resets the count for the next
      // launch (a replay of this one in a CUDA graph included)
      const unsigned long long old = atomicAdd(word, 1ull);
      if (static_cast<uint32_t>(old) + 1u == 2u * nblocks) atomicExch(word, tagged);
    } else {
      report(status, MOE_ERR_TIMEOUT);
    }
    __threadfence();
    ok_flag = ok ? 1 : 0;
  }
  __syncthreads();
  return ok_flag != 0;
}

// Rank of each lane's slot (expert e, or -1 for none) among the warp's slots
// so far of the same expert: the lanes hold 32 consecutive slots in order,
// `wc` the warp's running count per expert.
__device__ __forceinline__ int warp_rank(int e, int32_t* wc, int lane) {
  const uint32_t peers = __match_any_sync(0xffffffffu, e);
  int before = 0;
  if (e >= 0) before = wc[e];
  __syncwarp();
  if (e >= 0 && lane == __ffs(peers) - 1) wc[e] = before + __popc(peers);
  __syncwarp();
  return before + __popc(peers & ((1u << lane) - 1u));
}

// ------------------------------------------------------------ top-K select
// The group's K largest keys, exactly, without K sequential arg-max rounds:
// each lane sorts its VPL keys (bitonic networks on chunks of L = K rounded
// up to a power of two, merged down to the lane's L largest), then the
// group's lanes merge their lists in log2(G) butterfly steps, after which
// every lane of the group holds the group's L largest keys in descending
// order.  Keys are distinct (the expert id is part of the key), so the
// selection, and therefore ids and w, are the same as by arg-max rounds.

// Compare-exchange: the larger key to a, the smaller to b.
__device__ __forceinline__ void ce_desc(uint64_t& a, uint64_t& b) {
  const bool swap = b > a;
  const uint64_t hi = swap ? b : a;
  const uint64_t lo = swap ? a : b;
  a = hi;
  b = lo;
}

// Bitonic sort of N keys (a power of two) into descending order.
template <int N>
__device__ __forceinline__ void sort_desc(uint64_t (&x)[N]) {
#pragma unroll
  for (int k = 2; k <= N; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int l = i ^ j;
        if (l > i) {
          if ((i & k) == 0) {
            ce_desc(x[i], x[l]);
          } else {
            ce_desc(x[l], x[i]);
          }
        }
      }
}

// a := the N largest keys of a and b (each sorted descending), descending.
// The element-wise larger of a and b reversed holds exactly those N keys as
// a bitonic sequence, which one bitonic merge sorts.
template <int N>
__device__ __forceinline__ void merge_top(uint64_t (&a)[N], const uint64_t (&b)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) a[i] = b[N - 1 - i] > a[i] ? b[N - 1 - i] : a[i];
#pragma unroll
  for (int j = N >> 1; j > 0; j >>= 1)
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((i & j) == 0) ce_desc(a[i], a[i | j]);
}

// Slots that phase 1 hands to phase 3 in registers: the lane's slot of each
// of the warp's first S passes (flat index j, expert e, rank in the warp r;
// j = -1 for none).  Later passes go through pos in memory.
template <int S>
struct HeldSlots {
  int j[S];
  int e[S];
  int r[S];
};

// Phase 1, shared by both kernels: the tokens [t0, t1) of one warp.  For
// each of them a group of G lanes selects the top-K keys and computes the
// routing weights (or, for given routing, the ids are read).  Each slot's
// rank among the warp's earlier slots of the same expert is kept for phase
// 3; `wc` is the warp's running count per expert.  VPL: keys per lane,
// L: sorted list length (K <= L <= VPL, powers of two, G * VPL >= E, G >= K).
// Returns the first flat slot whose rank went to pos in memory.
template <int VPL, int L, int S>
__device__ __forceinline__ long select_slots(const float* __restrict__ logits,
                                             const float* __restrict__ bias, int mode,
                                             int32_t* __restrict__ ids, float* __restrict__ w,
                                             int32_t* __restrict__ pos, int32_t* wc, long t0,
                                             long t1, int E, int K, int G, int lane,
                                             int32_t* status, HeldSlots<S>& held) {
#pragma unroll
  for (int s = 0; s < S; ++s) {
    held.j[s] = -1;
    held.e[s] = -1;
    held.r[s] = 0;
  }
  // keep slot (j, e, r) of pass s in registers, or its rank in pos
  auto keep = [&](int s, long j, int e, int r) {
    if (s < S) {
#pragma unroll
      for (int q = 0; q < S; ++q)
        if (q == s) {
          held.j[q] = e >= 0 ? static_cast<int>(j) : -1;
          held.e[q] = e;
          held.r[q] = r;
        }
    } else if (e >= 0) {
      pos[j] = r;
    }
  };
  if (mode == MOE_SCORE_GIVEN) {
    int s = 0;
    for (long jb = t0 * K; jb < t1 * K; jb += 32, ++s) {
      const long j = jb + lane;
      int e = -1;
      if (j < t1 * K) {
        e = ids[j];
        if (e < 0 || e >= E) {
          report(status, MOE_ERR_DEVICE);
          pos[j] = -1;
          e = -1;
        }
      }
      keep(s, j, e, warp_rank(e, wc, lane));
    }
    return min(t1 * K, t0 * K + 32L * S);
  }
  const int gl = lane & (G - 1);  // lane within the token's group
  const int gbase = lane - gl;    // first lane of the group
  const int tpp = 32 / G;         // tokens per pass of the warp
  int s = 0;
  for (long tb = t0; tb < t1; tb += tpp, ++s) {  // the same trip count in every lane
    const long t = tb + lane / G;
    const bool live = t < t1;
    // all of the lane's scores are loaded before any is used
    float sv[VPL], bv[VPL];
    const float* row = logits + t * E;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = gl + G * i;
      const bool ok = live && e < E;
      sv[i] = ok ? __ldg(row + e) : 0.f;
      bv[i] = (ok && bias != nullptr) ? __ldg(bias + e) : 0.f;
    }
    asm volatile("" ::: "memory");
    uint64_t top[L];
#pragma unroll
    for (int c = 0; c < VPL / L; ++c) {
      uint64_t part[L];
#pragma unroll
      for (int q = 0; q < L; ++q) {
        const int i = c * L + q;
        const int e = gl + G * i;
        part[q] = (live && e < E)
                      ? score_key(bias != nullptr ? __fadd_rn(sv[i], bv[i]) : sv[i], e)
                      : 0ull;
      }
      sort_desc<L>(part);
      if (c == 0) {
#pragma unroll
        for (int q = 0; q < L; ++q) top[q] = part[q];
      } else {
        merge_top<L>(top, part);
      }
    }
    for (int off = G >> 1; off > 0; off >>= 1) {
      uint64_t other[L];
#pragma unroll
      for (int q = 0; q < L; ++q) other[q] = __shfl_xor_sync(0xffffffffu, top[q], off);
      merge_top<L>(top, other);
    }
    uint64_t mine = 0;  // group lane k takes slot k
#pragma unroll
    for (int q = 0; q < L; ++q) mine = (gl == q) ? top[q] : mine;
    const float my_v = key_score(mine);
    const int my_e = key_expert(mine);
    // routing weights of the K selected scores; slot 0 holds the largest
    float ex = 0.f;
    if (mode == MOE_SCORE_SOFTMAX_TOPK) {
      const float m = key_score(top[0]);
      if (gl < K) ex = expf(my_v - m);
    } else {
      if (gl < K) ex = 1.0f / (1.0f + expf(-my_v));
    }
    float sum = 0.f;  // ascending slot order
    for (int k = 0; k < K; ++k) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, ex, gbase + k));
    int e = -1;
    const long j = t * K + gl;
    if (live && gl < K) {
      ids[j] = my_e;
      w[j] = __fdiv_rn(ex, sum);
      e = my_e;
    }
    // the lanes hold the pass's slots in flat order (token, then slot)
    keep(s, j, e, warp_rank(e, wc, lane));
  }
  return min(t1, t0 + static_cast<long>(tpp) * S) * K;
}

// Phases 2 (its end) and 3, shared by both kernels.  In shared memory: tot
// (every block's slots per expert summed: group_sizes) and pre (the blocks
// before this one).  group_offsets is the exclusive scan of tot over the
// experts (thread i holds `per` consecutive ones); then
// pos = group_offsets[e] + pre[e] + the warp's prefix + its rank in the
// warp, the stable order in the flat slot index t*K+k, and row_src[pos] = j.
// Rows that no valid slot fills (only when some id was out of range) get -1.
struct PlaceCtx {
  const int32_t* tot;
  const int32_t* pre;
  int32_t* basev;
  int32_t* wsum;  // [32]
  int* filled;
  int block, nblocks;
};

template <int S>
__device__ __forceinline__ void place_slots(const PlaceCtx& c, const int32_t* wc,
                                            const HeldSlots<S>& held, long jmem0,
                                            const int32_t* __restrict__ ids,
                                            int32_t* __restrict__ pos,
                                            int32_t* __restrict__ row_src,
                                            int32_t* __restrict__ group_sizes,
                                            int32_t* __restrict__ group_offsets, long t1, int T,
                                            int E, int K) {
  const int NT = static_cast<int>(blockDim.x);
  const int WARPS = NT >> 5;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (E + NT - 1) / NT;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += c.tot[e];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) c.wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < WARPS ? c.wsum[lane] : 0;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += u;
    }
    if (lane < WARPS) c.wsum[lane] = x - v;
  }
  __syncthreads();
  int run = c.wsum[warp] + incl - local;
  for (int e = e0; e < e1; ++e) {
    c.basev[e] = run + c.pre[e];
    if (c.block == 0) {
      group_sizes[e] = c.tot[e];
      group_offsets[e] = run;
    }
    run += c.tot[e];
  }
  if (e0 < e1 && e1 == E) {
    *c.filled = run;
    if (c.block == 0) group_offsets[E] = run;
  }
  __syncthreads();
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int j = held.j[s];
    if (j < 0) continue;
    const int e = held.e[s];
    const int p = c.basev[e] + wc[e] + held.r[s];
    pos[j] = p;
    row_src[p] = j;
  }
  for (long j = jmem0 + lane; j < t1 * K; j += 32) {
    const int e = ids[j];
    if (e < 0 || e >= E) continue;  // dropped slot: pos is already -1
    const int p = c.basev[e] + wc[e] + pos[j];
    pos[j] = p;
    row_src[p] = static_cast<int32_t>(j);
  }
  const long R = static_cast<long>(T) * K;
  for (long r = *c.filled + static_cast<long>(c.block) * NT + tid; r < R;
       r += static_cast<long>(c.nblocks) * NT)
    row_src[r] = -1;
}

// Passes per warp whose slots phase 1 hands to phase 3 in registers.
constexpr int kHeldPasses = 2;

// Each warp zeroes its own row of per-warp counts (no other warp reads it
// before the block's barrier after phase 1).
__device__ __forceinline__ void zero_row(int32_t* wc, int E, int lane) {
  for (int e = lane; e < E; e += 32) wc[e] = 0;
  __syncwarp();
}

// The cooperative kernel (any number of tokens): WARPS = blockDim.x / 32
// warps per block (at most kRouteMaxWarps), each owning `tpw` consecutive
// tokens.  Shared memory: per-warp counts [WARPS][E], then tot, pre and
// basev [E] each, then the per-run partial sums [max(32 * WARPS, E)] twice.
// Global scratch: the barrier word and the blocks' totals [blocks][E].
template <int VPL, int L>
__global__ void __launch_bounds__(kRouteMaxWarps * 32, 1) route_kernel(
    const float* __restrict__ logits, const float* __restrict__ bias, int mode,
    int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ group_sizes,
    int32_t* __restrict__ group_offsets, int32_t* __restrict__ pos,
    int32_t* __restrict__ row_src, unsigned long long* bar, int32_t* counts, int T, int E, int K,
    int G, int tpw, int32_t* status, uint64_t limit_ns) {
  const int NT = static_cast<int>(blockDim.x);
  const int WARPS = NT >> 5;
  extern __shared__ int32_t sm[];
  int32_t* wcnt = sm;               // [WARPS][E]
  int32_t* tot = sm + WARPS * E;    // [E]
  int32_t* pre = tot + E;           // [E]
  int32_t* basev = pre + E;         // [E]
  int32_t* part_tot = basev + E;    // [max(NT, E)]
  int32_t* part_pre = part_tot + (NT > E ? NT : E);
  __shared__ int32_t wsum[32];
  __shared__ int s_filled;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* wc = wcnt + warp * E;
  zero_row(wc, E, lane);
  const long t0 = min(static_cast<long>(T), (static_cast<long>(blockIdx.x) * WARPS + warp) * tpw);
  const long t1 = min(static_cast<long>(T), t0 + tpw);

  HeldSlots<kHeldPasses> held;
  const long jmem0 = select_slots<VPL, L, kHeldPasses>(logits, bias, mode, ids, w, pos, wc, t0,
                                                       t1, E, K, G, lane, status, held);
  __syncthreads();
  // per-warp counts -> exclusive prefixes over the block's warps; totals out
  for (int e = tid; e < E; e += NT) {
    int run = 0;
    for (int q = 0; q < WARPS; ++q) {
      const int v = wcnt[q * E + e];
      wcnt[q * E + e] = run;
      run += v;
    }
    counts[static_cast<long>(blockIdx.x) * E + e] = run;
  }
  const int nb = static_cast<int>(gridDim.x);
  if (!grid_barrier(bar, static_cast<uint32_t>(nb), status, limit_ns)) return;

  // The blocks' totals per expert summed before this block (its prefix) and
  // over all blocks (group_sizes).  Thread (g, e) sums expert e over the g-th
  // of S runs of blocks, threads indexed by expert so that loads coalesce and
  // with several independent loads in flight; the runs' sums then meet in
  // shared memory.
  {
    const int S = max(1, NT / E);
    const int self = static_cast<int>(blockIdx.x);
    const int per_run = (nb + S - 1) / S;
    for (int i = tid; i < S * E; i += NT) {
      const int g = i / E, e = i - g * E;
      const int q0 = min(nb, g * per_run), q1 = min(nb, q0 + per_run);
      int p = 0, sum = 0;
#pragma unroll 8
      for (int q = q0; q < q1; ++q) {
        const int v = __ldcg(counts + static_cast<long>(q) * E + e);
        sum += v;
        p += (q < self) ? v : 0;
      }
      part_tot[i] = sum;
      part_pre[i] = p;
    }
    __syncthreads();
    for (int e = tid; e < E; e += NT) {
      int p = 0, sum = 0;
      for (int g = 0; g < S; ++g) {
        sum += part_tot[g * E + e];
        p += part_pre[g * E + e];
      }
      tot[e] = sum;
      pre[e] = p;
    }
  }
  __syncthreads();
  const PlaceCtx c{tot, pre, basev, wsum, &s_filled, static_cast<int>(blockIdx.x), nb};
  place_slots(c, wc, held, jmem0, ids, pos, row_src, group_sizes, group_offsets, t1, T, E, K);
}

// The cluster kernel (few tokens): the grid is one thread-block cluster of
// at most kRouteMaxCluster blocks.  Each block writes its totals straight
// into every block's shared memory and the blocks meet at the hardware
// cluster barrier; there is no global scratch, no cooperative launch and no
// read of other blocks' totals through memory, whose fixed costs are most
// of the time when tokens are few.  Blocks of kRouteMaxWarps warps; shared
// memory: per-warp counts [WARPS][E], then tot, pre and basev [E] each,
// then every block's totals [kRouteMaxCluster][E].
constexpr int kRouteMaxCluster = 16;

template <int VPL, int L>
__global__ void __launch_bounds__(kRouteMaxWarps * 32, 1) route_cluster_kernel(
    const float* __restrict__ logits, const float* __restrict__ bias, int mode,
    int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ group_sizes,
    int32_t* __restrict__ group_offsets, int32_t* __restrict__ pos,
    int32_t* __restrict__ row_src, int T, int E, int K, int G, int tpw, int32_t* status) {
  const int NT = static_cast<int>(blockDim.x);
  const int WARPS = NT >> 5;
  extern __shared__ int32_t sm[];
  int32_t* wcnt = sm;               // [WARPS][E]
  int32_t* tot = sm + WARPS * E;    // [E]
  int32_t* pre = tot + E;           // [E]
  int32_t* basev = pre + E;         // [E]
  int32_t* all = basev + E;         // [kRouteMaxCluster][E]
  __shared__ int32_t wsum[32];
  __shared__ int s_filled;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = static_cast<int>(cluster_ctarank());
  const int nb = static_cast<int>(gridDim.x);  // the grid is the cluster
  cluster_arrive_release();  // this block has started (waited for before the tables are written)
  int32_t* wc = wcnt + warp * E;
  zero_row(wc, E, lane);
  const long t0 = min(static_cast<long>(T), (static_cast<long>(rank) * WARPS + warp) * tpw);
  const long t1 = min(static_cast<long>(T), t0 + tpw);

  HeldSlots<kHeldPasses> held;
  const long jmem0 = select_slots<VPL, L, kHeldPasses>(logits, bias, mode, ids, w, pos, wc, t0,
                                                       t1, E, K, G, lane, status, held);
  __syncthreads();
  cluster_wait_acquire();  // every block has started: its table may be written
  // per-warp counts -> exclusive prefixes over the block's warps; the
  // block's totals into row `rank` of every block's table
  for (int e = tid; e < E; e += NT) {
    int run = 0;
    for (int q = 0; q < WARPS; ++q) {
      const int v = wcnt[q * E + e];
      wcnt[q * E + e] = run;
      run += v;
    }
    const uint32_t a = smem_u32(all + rank * E + e);
    for (int q = 0; q < nb; ++q) st_cluster_u32(mapa_shared(a, static_cast<uint32_t>(q)), run);
  }
  cluster_sync();  // every block's totals are in every block's table
  for (int e = tid; e < E; e += NT) {
    int p = 0, sum = 0;
    for (int q = 0; q < nb; ++q) {
      const int v = all[q * E + e];
      sum += v;
      p += (q < rank) ? v : 0;
    }
    tot[e] = sum;
    pre[e] = p;
  }
  __syncthreads();
  const PlaceCtx c{tot, pre, basev, wsum, &s_filled, rank, nb};
  place_slots(c, wc, held, jmem0, ids, pos, row_src, group_sizes, group_offsets, t1, T, E, K);
}

size_t route_smem_bytes(int warps, int E) {
  const size_t part = static_cast<size_t>(32 * warps > E ? 32 * warps : E);
  return (static_cast<size_t>(warps + 3) * static_cast<size_t>(E) + 2 * part) * sizeof(int32_t);
}

// A block's warps each own a run of tokens; with few tokens it is the
// latency of one pass of the top-K that counts, so blocks start at 8 warps
// (2 per scheduler) to spread the passes over the SMs, and grow to
// kRouteMaxWarps warps when there are more passes than that covers.  Blocks
// stay at 8 warps or more because after the barrier each block reads every
// block's totals, (blocks * E) / (threads per block) loads per thread.
template <int VPL, int L>
cudaError_t launch_route(const float* logits, const float* bias, int mode, int32_t* ids, float* w,
                         int32_t* group_sizes, int32_t* group_offsets, int32_t* pos,
                         int32_t* row_src, int32_t* dev_status, unsigned long long* bar,
                         int32_t* counts, long max_blocks, const moe_dims& d, int G,
                         cudaStream_t s) {
  auto kern = route_kernel<VPL, L>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  // the shared-memory opt-in (for the largest block and E) once per device,
  // and the blocks of that size one SM holds (a bound for smaller ones)
  static std::atomic<int> per_sm[64];
  int bps = per_sm[dev].load(std::memory_order_acquire);
  if (bps == 0) {
    const size_t smax = route_smem_bytes(kRouteMaxWarps, 1024);
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smax));
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, kRouteMaxWarps * 32, smax);
    if (err != cudaSuccess) return err;
    if (bps < 1) return cudaErrorInvalidConfiguration;
    per_sm[dev].store(bps, std::memory_order_release);
  }
  const int sms = sm_count();
  const int tpp = 32 / G;  // tokens per warp pass
  const long passes = (d.T + tpp - 1) / tpp;
  int warps = 8;
  while (warps < kRouteMaxWarps && (passes + warps - 1) / warps > sms) warps <<= 1;
  // at most one block per SM: every block reads every block's totals after
  // the barrier, so the grid is kept about as wide as the machine, not wider
  long blocks = (passes + warps - 1) / warps;
  long resident = static_cast<long>(bps) * sms;
  if (resident > sms) resident = sms;
  if (blocks > resident) blocks = resident;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  // tokens per warp: a whole number of passes, the fewest that cover T
  long tpw = (d.T + blocks * warps - 1) / (blocks * warps);
  tpw = (tpw + tpp - 1) / tpp * tpp;
  blocks = (d.T + static_cast<long>(warps) * tpw - 1) / (static_cast<long>(warps) * tpw);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(warps * 32), 1, 1);
  cfg.dynamicSmemBytes = route_smem_bytes(warps, d.E);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, logits, bias, mode, ids, w, group_sizes, group_offsets,
                            pos, row_src, bar, counts, d.T, d.E, d.K, G,
                            static_cast<int>(tpw),
                            dev_status, kDefaultWaitLimitNs);
}

size_t route_cluster_smem_bytes(int warps, int E) {
  return static_cast<size_t>(warps + 3 + kRouteMaxCluster) * static_cast<size_t>(E) *
         sizeof(int32_t);
}

// Blocks of the routing cluster: 16 (a non-portable cluster size) where the
// device can hold one such cluster of these blocks, else 8, else 0 (the
// cluster kernel is not used).  Found once per device and instantiation.
template <int VPL, int L>
int route_cluster_blocks(int dev) {
  static std::atomic<int> found[64];  // 0: not yet known; -1: no cluster
  int c = found[dev].load(std::memory_order_acquire);
  if (c != 0) return c > 0 ? c : 0;
  auto kern = route_cluster_kernel<VPL, L>;
  const size_t smax = route_cluster_smem_bytes(kRouteMaxWarps, 1024);
  c = -1;
  bool refused = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smax)) != cudaSuccess;
  if (!refused) {
    refused = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
              cudaSuccess;
    for (int want = refused ? 8 : kRouteMaxCluster; want >= 8; want >>= 1) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(want);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(static_cast<unsigned>(want), 1, 1);
      cfg.blockDim = dim3(kRouteMaxWarps * 32, 1, 1);
      cfg.dynamicSmemBytes = smax;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        refused = true;
      } else if (n >= 1) {
        c = want;
        break;
      }
    }
  }
  if (refused) (void)cudaGetLastError();  // a size the device refuses leaves no error behind
  found[dev].store(c, std::memory_order_release);
  return c > 0 ? c : 0;
}

// One cluster of C blocks; every warp owns a whole number of the passes
// that cover T.
template <int VPL, int L>
cudaError_t launch_route_cluster(const float* logits, const float* bias, int mode, int32_t* ids,
                                 float* w, int32_t* group_sizes, int32_t* group_offsets,
                                 int32_t* pos, int32_t* row_src, int32_t* dev_status, int C,
                                 const moe_dims& d, int G, cudaStream_t s) {
  const int warps = kRouteMaxWarps;
  const int tpp = 32 / G;
  long tpw = (d.T + static_cast<long>(C) * warps - 1) / (static_cast<long>(C) * warps);
  tpw = (tpw + tpp - 1) / tpp * tpp;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(C), 1, 1);
  cfg.blockDim = dim3(warps * 32, 1, 1);
  cfg.dynamicSmemBytes = route_cluster_smem_bytes(warps, d.E);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_cluster_kernel<VPL, L>, logits, bias, mode, ids, w,
                            group_sizes, group_offsets, pos, row_src, d.T, d.E, d.K, G,
                            static_cast<int>(tpw), dev_status);
}

// The cluster kernel while each of its warps has no more passes than phase
// 1 hands over in registers and the selection is light (given routing, or
// E <= 64); the cooperative kernel otherwise.  Measured on GB300 (one launch
// behind a busy kernel, us, cluster / cooperative): given routing at 1024
// tokens 8.4 / 9.9; E = 8, K = 2 at 256 tokens 9.8 / 11.9; E = 64, K = 4
// at 1024 tokens 11.8 / 13.0; but E = 128, K = 8 at 256 tokens 13.9 / 12.9
// and at 1024 tokens 14.4 / 13.9: there the top-K of 16 SMs is the larger
// cost than the cooperative grid's barrier and exchange.
template <int VPL, int L>
cudaError_t launch_route_any(const float* logits, const float* bias, int mode, int32_t* ids,
                             float* w, int32_t* group_sizes, int32_t* group_offsets, int32_t* pos,
                             int32_t* row_src, int32_t* dev_status, unsigned long long* bar,
                             int32_t* counts, long max_blocks, const moe_dims& d, int G,
                             cudaStream_t s) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int C = route_cluster_blocks<VPL, L>(dev);
  if (C > 0 && (mode == MOE_SCORE_GIVEN || d.E <= 64)) {
    // tokens per warp as the cluster launch sets it, and that warp's passes
    const long tpp = 32 / G;
    const long cw = static_cast<long>(C) * kRouteMaxWarps;
    const long tpw = ((d.T + cw - 1) / cw + tpp - 1) / tpp * tpp;
    const long passes = (mode == MOE_SCORE_GIVEN) ? (tpw * d.K + 31) / 32 : tpw / tpp;
    if (passes <= kHeldPasses)
      return launch_route_cluster<VPL, L>(logits, bias, mode, ids, w, group_sizes, group_offsets,
                                          pos, row_src, dev_status, C, d, G, s);
  }
  return launch_route<VPL, L>(logits, bias, mode, ids, w, group_sizes, group_offsets, pos, row_src,
                           dev_status, bar, counts, max_blocks, d, G, s);
}

// Scratch of moe_route_histogram_noalloc: the barrier counter (first 256
// bytes) and the per-block expert totals live in this fixed array instead
// of a caller workspace.  Every GPU that loads the library holds it (1 MiB)
// until the process exits.
static __device__ __align__(256) int32_t g_route_scratch[kRouteStaticScratchInts];

}  // namespace

cudaError_t launch_route_histogram(const float* logits, const float* bias, int mode, int32_t* ids,
                                   float* w, int32_t* group_sizes, int32_t* group_offsets,
                                   int32_t* pos, int32_t* row_src, int32_t* dev_status,
                                   void* scratch, long max_blocks, const moe_dims& d,
                                   cudaStream_t s) {
  if (d.T == 0) {
    cudaError_t err = cudaMemsetAsync(group_sizes, 0, static_cast<size_t>(d.E) * 4, s);
    if (err != cudaSuccess) return err;
    return cudaMemsetAsync(group_offsets, 0, static_cast<size_t>(d.E + 1) * 4, s);
  }
  // the barrier word at byte 64: the GEMMs keep their tile counter at byte 0
  // of the same workspace
  auto* bar = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(scratch) + 64);
  int32_t* counts = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(scratch) + kRouteBarrierBytes);
  // L: K rounded up to a power of two (at least 2).  G lanes per token, a
  // power of two >= K, with VPL keys each (VPL >= L, at least 4, G * VPL >=
  // E): the fewest keys per lane that cover E, the lanes doubled while a
  // lane would hold more than 16 keys
  int L = 2;
  while (L < d.K) L <<= 1;
  int G = 1;
  while (G < d.K) G <<= 1;
  int vpl = 4;
  while (vpl < L || G * vpl < d.E) vpl <<= 1;
  while (vpl > 16 && G < 32 && vpl / 2 >= L) {
    G <<= 1;
    vpl >>= 1;
  }
#define MOE_ROUTE(V, LL)                                                                   \
  launch_route_any<V, LL>(logits, bias, mode, ids, w, group_sizes, group_offsets, pos,   \
                          row_src, dev_status, bar, counts, max_blocks, d, G, s)
  switch (vpl * 64 + L) {
    case 4 * 64 + 2: return MOE_ROUTE(4, 2);
    case 4 * 64 + 4: return MOE_ROUTE(4, 4);
    case 8 * 64 + 2: return MOE_ROUTE(8, 2);
    case 8 * 64 + 4: return MOE_ROUTE(8, 4);
    case 8 * 64 + 8: return MOE_ROUTE(8, 8);
    case 16 * 64 + 2: return MOE_ROUTE(16, 2);
    case 16 * 64 + 4: return MOE_ROUTE(16, 4);
    case 16 * 64 + 8: return MOE_ROUTE(16, 8);
    case 16 * 64 + 16: return MOE_ROUTE(16, 16);
    case 32 * 64 + 2: return MOE_ROUTE(32, 2);
    case 32 * 64 + 4: return MOE_ROUTE(32, 4);
    case 32 * 64 + 8: return MOE_ROUTE(32, 8);
    case 32 * 64 + 16: return MOE_ROUTE(32, 16);
    default: return MOE_ROUTE(32, 32);
  }
#undef MOE_ROUTE
}

// Unique id of the calling thread's current CUDA context (never reused
// within a process), or 0 when there is none or the driver cannot say.
static unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// The same three kernels with their scratch in g_route_scratch.  The host
// only knows a stand-in for the array's name; its device address is looked
// up (with the device current) on the first call on each device, and again
// whenever the device's context has changed since (after a cudaDeviceReset
// the array lives at a new address in the new context).
cudaError_t launch_route_histogram_static(const float* logits, const float* bias, int mode,
                                          int32_t* ids, float* w, int32_t* group_sizes,
                                          int32_t* group_offsets, int32_t* pos, int32_t* row_src,
                                          int32_t* dev_status, const moe_dims& d,
                                          cudaStream_t s) {
  struct Cached {
    int32_t* ptr;
    unsigned long long ctx;
  };
  static std::mutex mu;
  static Cached scratch_of_device[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int32_t* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    Cached& c = scratch_of_device[dev];
    const unsigned long long ctx = current_context_id();
    if (c.ptr == nullptr || ctx == 0 || ctx != c.ctx) {
      err = cudaGetSymbolAddress((void**)&ptr, g_route_scratch);
      if (err != cudaSuccess) return err;
      c.ptr = ptr;
      c.ctx = current_context_id();  // the lookup made the device's context current
    }
    ptr = c.ptr;
  }
  // the barrier word, then the totals of at most max_blocks blocks
  const long max_blocks =
      static_cast<long>((kRouteStaticScratchInts - kRouteBarrierBytes / sizeof(int32_t)) /
                        static_cast<size_t>(d.E));
  // the kernel writes every total it reads, and every launch leaves the
  // barrier word ready for the next, so nothing left by an earlier call leaks
  return launch_route_histogram(logits, bias, mode, ids, w, group_sizes, group_offsets, pos,
                                row_src, dev_status, ptr, max_blocks, d, s);
}

}  // namespace moe
