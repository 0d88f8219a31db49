// Routing and group_size histogram of the MoE block.
//
// MaxText "Gemma4 26B MoE on TPU v6e: MaxText layer/model optimizations",
// Commits table row 6: top_k_weights and group_size are computed next to the
// rest of the block; MaxText "MoE: fused TensorCore Pallas permute/combine
// kernels and split-expert wi layout for TPU v6e", Commits table row 2: the
// group_size histogram is computed before the token gather.
//
// Three kernels, all deterministic (no atomic decides an order; atomics only
// add up counts):
//   1. route_topk: one group of G lanes per token (32/G tokens per warp,
//      grid-stride over all tokens) selects the top-K scores by K rounds of
//      a group-wide (score desc, id asc) arg-max, computes the routing
//      weights, and adds each slot to the count of its (chunk of 256
//      tokens, expert) pair in global memory.
//   2. route_scan: per expert, the exclusive prefix of the counts over
//      chunks, group_sizes, and the exclusive prefix over experts
//      (group_offsets); threads are indexed by expert so reads coalesce.
//   3. route_rank: per chunk, each warp ranks its contiguous run of slots
//      with __match_any_sync; pos = group_offsets[e] + chunk prefix + warp
//      prefix + rank, i.e. the stable order in the flat slot index t*K+k.
#include <cuda.h>

#include <cfloat>
#include <climits>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;  // 8 warps
constexpr int kRouteWarps = kRouteThreads / 32;

__device__ __forceinline__ bool better(float v1, int e1, float v2, int e2) {
  return v1 > v2 || (v1 == v2 && e1 < e2);
}

// One group of G lanes per token (G a power of two, G >= K, G * VPL >= E):
// a warp selects the top-K of 32/G tokens at once.  Lane i of a group holds
// the scores of experts i, i+G, i+2G, ...; each of the K rounds takes the
// group-wide (score desc, id asc) arg-max over the experts not yet taken, so
// slot k is the k-th largest score.
template <int VPL>
__global__ void __launch_bounds__(kRouteThreads) route_topk(
    const float* __restrict__ logits, const float* __restrict__ bias, int mode,
    int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ counts, int T, int E,
    int K, int G, int32_t* status) {
  const int lane = threadIdx.x & 31;
  if (mode == MOE_SCORE_GIVEN) {
    const long R = static_cast<long>(T) * K;
    for (long j = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; j < R;
         j += static_cast<long>(gridDim.x) * blockDim.x) {
      const int e = ids[j];
      const int chunk = static_cast<int>(j / K) / kRouteTokensPerChunk;
      if (e >= 0 && e < E) atomicAdd(&counts[static_cast<long>(chunk) * E + e], 1);
      else report(status, MOE_ERR_DEVICE);
    }
    return;
  }
  const int gl = lane & (G - 1);   // lane within the group
  const int gbase = lane - gl;     // first lane of the group
  const int groups_per_warp = 32 / G;
  const long groups_total = static_cast<long>(gridDim.x) * kRouteWarps * groups_per_warp;
  const long first = (static_cast<long>(blockIdx.x) * kRouteWarps + (threadIdx.x >> 5)) *
                         groups_per_warp + (lane / G);
  // every lane of a warp runs the same number of iterations (shuffles stay converged)
  const long warp_first = first - lane / G;
  for (long base = warp_first; base < T; base += groups_total) {
    const long t = base + lane / G;
    const bool live = t < T;
    float s[VPL];
    const float* row = logits + t * E;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = gl + G * i;
      if (live && e < E) {
        float v = __ldg(row + e);
        if (bias != nullptr) v = __fadd_rn(v, __ldg(bias + e));
        s[i] = v;
      } else {
        s[i] = -FLT_MAX;
      }
    }
    uint32_t taken = 0;
    float my_v = 0.f;
    int my_e = 0;
    for (int k = 0; k < K; ++k) {
      float bv = -FLT_MAX;
      int be = INT_MAX;  // "no candidate" loses to every real expert
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = gl + G * i;
        if (e < E && !((taken >> i) & 1u) && better(s[i], e, bv, be)) { bv = s[i]; be = e; }
      }
      for (int off = G >> 1; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (better(ov, oe, bv, be)) { bv = ov; be = oe; }
      }
      if (be != INT_MAX && (be & (G - 1)) == gl) taken |= 1u << (be / G);
      if (gl == k) { my_v = bv; my_e = be; }
    }
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
    if (live && gl < K) {
      const long j = t * K + gl;
      ids[j] = my_e;
      w[j] = __fdiv_rn(ex, sum);
      atomicAdd(&counts[(t / kRouteTokensPerChunk) * E + my_e], 1);
    }
  }
}

// One block of 1024 threads.  Thread (g, e) = (tid / E, tid % E) covers
// expert e over chunk group g (a contiguous run of chunks), so that each
// load of counts[c, 0..E) is coalesced across the threads of a group.
__global__ void __launch_bounds__(1024) route_scan(const int32_t* __restrict__ counts,
                                                   int32_t* __restrict__ chunk_excl, int nchunks,
                                                   int E, int32_t* __restrict__ group_sizes,
                                                   int32_t* __restrict__ group_offsets) {
  __shared__ int32_t part[1024];
  __shared__ int32_t tot[1024];
  __shared__ int32_t warp_sum[32];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int G = max(1, 1024 / E);
  const int e = tid % E, g = tid / E;
  const bool active = g < G;
  const int cpg = (nchunks + G - 1) / G;
  const int c0 = min(nchunks, g * cpg), c1 = min(nchunks, c0 + cpg);
  if (active) {
    int local = 0;
#pragma unroll 4
    for (int c = c0; c < c1; ++c) local += counts[static_cast<long>(c) * E + e];
    part[g * E + e] = local;
  }
  __syncthreads();
  if (tid < E) {
    int run = 0;
    for (int q = 0; q < G; ++q) {
      const int v = part[q * E + tid];
      part[q * E + tid] = run;
      run += v;
    }
    tot[tid] = run;
    group_sizes[tid] = run;
  }
  __syncthreads();
  // exclusive scan of tot[0..E) over the block
  const int v = (tid < E) ? tot[tid] : 0;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int ws = warp_sum[lane];
    int wi = ws;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += u;
    }
    warp_sum[lane] = wi - ws;
  }
  __syncthreads();
  const int excl = warp_sum[warp] + incl - v;
  if (tid < E) group_offsets[tid] = excl;
  if (tid == E - 1) group_offsets[E] = excl + v;
  if (active) {
    int run = part[g * E + e];
#pragma unroll 4
    for (int c = c0; c < c1; ++c) {
      const long idx = static_cast<long>(c) * E + e;
      const int cv = counts[idx];
      chunk_excl[idx] = run;
      run += cv;
    }
  }
}

// One block per chunk; warp w ranks slots [j0 + w*32K, j0 + (w+1)*32K).
__global__ void __launch_bounds__(kRouteThreads) route_rank(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ chunk_excl,
    const int32_t* __restrict__ group_offsets, int32_t* __restrict__ pos,
    int32_t* __restrict__ row_src, int T, int K, int E) {
  extern __shared__ int32_t sm[];
  int32_t* wrun = sm;                      // [kRouteWarps][E]
  int32_t* base = sm + kRouteWarps * E;    // [E]
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const long R = static_cast<long>(T) * K;
  // rows that no valid slot fills (only when some id was out of range)
  const long filled = group_offsets[E];
  for (long r = filled + static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; r < R;
       r += static_cast<long>(gridDim.x) * blockDim.x)
    row_src[r] = -1;

  for (int i = threadIdx.x; i < kRouteWarps * E; i += blockDim.x) wrun[i] = 0;
  __syncthreads();
  const long chunk_j0 = static_cast<long>(blockIdx.x) * kRouteTokensPerChunk * K;
  const long per_warp = 32L * K;
  const long j0 = chunk_j0 + warp * per_warp;
  const long j1 = min(R, j0 + per_warp);
  for (long j = j0 + lane; j < j1; j += 32) {
    const int e = ids[j];
    if (e >= 0 && e < E) atomicAdd(&wrun[warp * E + e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int v = wrun[w * E + e];
      wrun[w * E + e] = run;
      run += v;
    }
    base[e] = group_offsets[e] + chunk_excl[static_cast<long>(blockIdx.x) * E + e];
  }
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (long jb = j0; jb < j1; jb += 32) {
    const long j = jb + lane;
    int e = (j < j1) ? ids[j] : -1;
    const bool valid = (e >= 0 && e < E);
    if (!valid) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int before = 0;
    if (valid) before = wrun[warp * E + e];
    __syncwarp();
    if (valid) {
      const int rank = __popc(peers & lt_mask);
      const int p = base[e] + before + rank;
      if (lane == __ffs(peers) - 1) wrun[warp * E + e] = before + __popc(peers);
      pos[j] = p;
      row_src[p] = static_cast<int32_t>(j);
    } else if (j < j1) {
      pos[j] = -1;
    }
    __syncwarp();
  }
}

template <int VPL>
cudaError_t launch_topk(const float* logits, const float* bias, int mode, int32_t* ids, float* w,
                        int32_t* counts, const moe_dims& d, int G, int32_t* status,
                        cudaStream_t s) {
  long blocks;
  if (mode == MOE_SCORE_GIVEN) {
    blocks = (static_cast<long>(d.T) * d.K + kRouteThreads - 1) / kRouteThreads;
  } else {
    const long tokens_per_block = static_cast<long>(kRouteWarps) * (32 / G);
    blocks = (d.T + tokens_per_block - 1) / tokens_per_block;
  }
  const long cap = static_cast<long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  route_topk<VPL><<<static_cast<int>(blocks), kRouteThreads, 0, s>>>(
      logits, bias, mode, ids, w, counts, d.T, d.E, d.K, G, status);
  return cudaGetLastError();
}

// Scratch of moe_route_histogram_noalloc: the per-chunk expert counts and
// their prefixes live in this fixed array instead of a caller workspace.
// Every GPU that loads the library holds it (1 MiB) until the process exits.
static __device__ __align__(256) int32_t g_route_scratch[kRouteStaticScratchInts];

}  // namespace

cudaError_t launch_route_histogram(const float* logits, const float* bias, int mode, int32_t* ids,
                                   float* w, int32_t* group_sizes, int32_t* group_offsets,
                                   int32_t* pos, int32_t* row_src, int32_t* dev_status,
                                   int32_t* counts, int32_t* chunk_excl, const moe_dims& d,
                                   cudaStream_t s) {
  const int nchunks = route_chunks(d.T);
  cudaError_t err = cudaSuccess;
  if (nchunks > 0) {
    err = cudaMemsetAsync(counts, 0, static_cast<size_t>(nchunks) * d.E * sizeof(int32_t), s);
    if (err != cudaSuccess) return err;
    // G lanes per token: a power of two with G >= K and G * VPL >= E, VPL <= 32
    int G = 1;
    while (G < d.K) G <<= 1;
    while (G * 32 < d.E) G <<= 1;
    int vpl = (d.E + G - 1) / G;
    if (vpl <= 4) err = launch_topk<4>(logits, bias, mode, ids, w, counts, d, G, dev_status, s);
    else if (vpl <= 8) err = launch_topk<8>(logits, bias, mode, ids, w, counts, d, G, dev_status, s);
    else if (vpl <= 16) err = launch_topk<16>(logits, bias, mode, ids, w, counts, d, G, dev_status, s);
    else err = launch_topk<32>(logits, bias, mode, ids, w, counts, d, G, dev_status, s);
    if (err != cudaSuccess) return err;
  }
  route_scan<<<1, 1024, 0, s>>>(counts, chunk_excl, nchunks, d.E, group_sizes, group_offsets);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (nchunks > 0) {
    const size_t smem = static_cast<size_t>(kRouteWarps + 1) * d.E * sizeof(int32_t);
    route_rank<<<nchunks, kRouteThreads, smem, s>>>(ids, chunk_excl, group_offsets, pos, row_src,
                                                    d.T, d.K, d.E);
    err = cudaGetLastError();
  }
  return err;
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
  const size_t per = static_cast<size_t>(route_chunks(d.T)) * static_cast<size_t>(d.E);
  if (2 * per > kRouteStaticScratchInts) return cudaErrorInvalidValue;
  // launch_route_histogram clears the counts it uses before counting, and
  // rewrites every prefix it reads, so nothing left by an earlier call leaks.
  return launch_route_histogram(logits, bias, mode, ids, w, group_sizes, group_offsets, pos,
                                row_src, dev_status, ptr, ptr + per, d, s);
}

}  // namespace moe
