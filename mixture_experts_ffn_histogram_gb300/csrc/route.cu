// Routing and group_size histogram of the MoE block.
//
// MaxText "Gemma4 26B MoE on TPU v6e: MaxText layer/model optimizations",
// Commits table row 6: top_k_weights and group_size are computed next to the
// rest of the block; MaxText "MoE: fused TensorCore Pallas permute/combine
// kernels and split-expert wi layout for TPU v6e", Commits table row 2: the
// group_size histogram is computed before the token gather.
//
// One cooperative kernel (every block resident at once), three phases
// separated by one grid-wide barrier; deterministic (no atomic decides an
// order):
//   1. Each warp owns a contiguous run of tokens.  For each of them a group
//      of G lanes selects the top-K scores by K rounds of a group-wide
//      (score desc, id asc) arg-max and computes the routing weights (or, for
//      given routing, reads the ids).  Each slot's rank among the warp's
//      earlier slots of the same expert (__match_any_sync over 32 slots at a
//      time, plus the warp's running count per expert in shared memory) is
//      stored in pos for now.  The block then turns the per-warp counts into
//      prefixes over its warps and publishes its per-expert totals.
//   2. After the barrier every block sums the published totals of the
//      blocks before it (its prefix per expert) and of all blocks
//      (group_sizes), and scans group_sizes over experts (group_offsets).
//   3. pos = group_offsets[e] + block prefix + warp prefix + rank in warp,
//      i.e. the stable order in the flat slot index t*K+k; row_src[pos] = j.
// The kernel is the only launch: the grid barrier's word needs no clearing.
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

// The routing kernel.  VPL: scores per lane (G lanes per token, G a power of
// two with G >= K and G * VPL >= E); WARPS = blockDim.x / 32 warps per
// block (at most kRouteMaxWarps).  Each warp owns `tpw` consecutive tokens.
// Shared memory: per-warp counts [WARPS][E], then totals, block prefixes and
// bases [E] each, then the per-run partial sums [max(32 * WARPS, E)] twice.
// Global scratch: the barrier word and the blocks' totals [blocks][E].
template <int VPL>
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
  for (int i = tid; i < WARPS * E; i += NT) wcnt[i] = 0;
  __syncthreads();
  int32_t* wc = wcnt + warp * E;
  const long t0 = min(static_cast<long>(T), (static_cast<long>(blockIdx.x) * WARPS + warp) * tpw);
  const long t1 = min(static_cast<long>(T), t0 + tpw);

  // ---------------------------------------------------------------- phase 1
  if (mode == MOE_SCORE_GIVEN) {
    for (long jb = t0 * K; jb < t1 * K; jb += 32) {
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
      const int r = warp_rank(e, wc, lane);
      if (e >= 0) pos[j] = r;
    }
  } else {
    const int gl = lane & (G - 1);  // lane within the token's group
    const int gbase = lane - gl;    // first lane of the group
    const int tpp = 32 / G;         // tokens per pass of the warp
    for (long tb = t0; tb < t1; tb += tpp) {  // the same trip count in every lane
      const long t = tb + lane / G;
      const bool live = t < t1;
      // all of the lane's scores are loaded before any is used: the compiler
      // would otherwise sink each load into the selection chain below and
      // pay one memory round trip per score (measured: ~10 us per pass at
      // E = 128)
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
      uint64_t key[VPL];
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = gl + G * i;
        key[i] = (live && e < E)
                     ? score_key(bias != nullptr ? __fadd_rn(sv[i], bv[i]) : sv[i], e)
                     : 0ull;
      }
      // round k takes the group's largest key below round k-1's: the k-th
      // largest score (ties: lower id first); within a lane as a max tree
      // (a short dependency chain), then across the group's lanes
      uint64_t last = ~0ull, mine = 0;
      for (int k = 0; k < K; ++k) {
        uint64_t c[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) c[i] = key[i] < last ? key[i] : 0ull;
#pragma unroll
        for (int w = VPL / 2; w > 0; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) c[i] = c[i + w] > c[i] ? c[i + w] : c[i];
        uint64_t best = c[0];
        for (int off = G >> 1; off > 0; off >>= 1) {
          const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
          best = o > best ? o : best;
        }
        last = best;
        if (gl == k) mine = best;
      }
      const float my_v = key_score(mine);
      const int my_e = key_expert(mine);
      // routing weights of the K selected scores (group lane k holds slot k)
      float ex = 0.f;
      if (mode == MOE_SCORE_SOFTMAX_TOPK) {
        const float m = __shfl_sync(0xffffffffu, my_v, gbase);
        if (gl < K) ex = expf(my_v - m);
      } else {
        if (gl < K) ex = 1.0f / (1.0f + expf(-my_v));
      }
      float sum = 0.f;  // ascending slot order
      for (int k = 0; k < K; ++k) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, ex, gbase + k));
      int e = -1;
      if (live && gl < K) {
        const long j = t * K + gl;
        ids[j] = my_e;
        w[j] = __fdiv_rn(ex, sum);
        e = my_e;
      }
      // the lanes hold the pass's slots in flat order (token, then slot)
      const int r = warp_rank(e, wc, lane);
      if (e >= 0) pos[t * K + gl] = r;
    }
  }
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

  // ---------------------------------------------------------------- phase 2
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
  // exclusive scan of tot over the experts: thread i holds `per` consecutive ones
  const int per = (E + NT - 1) / NT;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += tot[e];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < WARPS ? wsum[lane] : 0;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += u;
    }
    if (lane < WARPS) wsum[lane] = x - v;
  }
  __syncthreads();
  int run = wsum[warp] + incl - local;
  for (int e = e0; e < e1; ++e) {
    basev[e] = run + pre[e];
    if (blockIdx.x == 0) {
      group_sizes[e] = tot[e];
      group_offsets[e] = run;
    }
    run += tot[e];
  }
  if (e0 < e1 && e1 == E) {
    s_filled = run;
    if (blockIdx.x == 0) group_offsets[E] = run;
  }
  __syncthreads();

  // ---------------------------------------------------------------- phase 3
  for (long j = t0 * K + lane; j < t1 * K; j += 32) {
    const int e = ids[j];
    if (e < 0 || e >= E) continue;  // dropped slot: pos is already -1
    const int p = basev[e] + wc[e] + pos[j];
    pos[j] = p;
    row_src[p] = static_cast<int32_t>(j);
  }
  // rows that no valid slot fills (only when some id was out of range)
  const long R = static_cast<long>(T) * K;
  for (long r = s_filled + static_cast<long>(blockIdx.x) * NT + tid; r < R;
       r += static_cast<long>(gridDim.x) * NT)
    row_src[r] = -1;
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
template <int VPL>
cudaError_t launch_route(const float* logits, const float* bias, int mode, int32_t* ids, float* w,
                         int32_t* group_sizes, int32_t* group_offsets, int32_t* pos,
                         int32_t* row_src, int32_t* dev_status, unsigned long long* bar,
                         int32_t* counts, long max_blocks, const moe_dims& d, int G,
                         cudaStream_t s) {
  auto kern = route_kernel<VPL>;
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
  // G lanes per token: a power of two with G >= K and G * VPL >= E, VPL <= 32
  int G = 1;
  while (G < d.K) G <<= 1;
  while (G * 32 < d.E) G <<= 1;
  const int vpl = (d.E + G - 1) / G;
#define MOE_ROUTE(V)                                                                     \
  launch_route<V>(logits, bias, mode, ids, w, group_sizes, group_offsets, pos, row_src, \
                  dev_status, bar, counts, max_blocks, d, G, s)
  if (vpl <= 4) return MOE_ROUTE(4);
  if (vpl <= 8) return MOE_ROUTE(8);
  if (vpl <= 16) return MOE_ROUTE(16);
  return MOE_ROUTE(32);
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
