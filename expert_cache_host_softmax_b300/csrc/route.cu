// route.cu -- router top-k + softmax, permute-by-expert, and the on-device
// LRU slot plan.
//
// "FreeToken: Run Frontier MoE Models on Your Own GPU, and the RAM It Takes",
// section "Why a Huge MoE Model Fits on One Consumer GPU": a router sends each
// token to a few experts.  The GPU keeps an LRU cache of expert slots, one
// global pool shared across layers.  A hit runs at GPU speed; a miss is
// streamed over PCIe.
//
// Readings where the page is silent: top-k on the raw logits, ties to the
// lower expert id; gates = softmax over the k selected logits.  A lookup is
// one distinct (layer, expert) per call.  Hits become most recent in
// ascending expert id.  Then misses, in ascending id, take the lowest free
// slot or the least recent slot.
//
// The recency list lives on the device as an array of slot ids, least recent
// first.  Free slots sit at the front in index order.  One call rewrites it
// in a single block-wide compaction:
//   [untouched non-victims in old order] [hits, ascending id] [misses, ascending id]
// The victims are the first n_miss non-hit entries of the old order.  So the
// whole LRU update is O(S / blockDim) per thread, plus two block scans.
#include <math.h>

#include <algorithm>

#include "ft_internal.cuh"

#include "route_dev.cuh"

namespace ftmoe {

namespace {

// ---------------------------------------------------------------- kernels

// Whole routing of a small call in one CTA (see route_body).
__global__ void __launch_bounds__(kRouteThreads) route_small_kernel(RouteArgs a) {
  extern __shared__ int smem[];
  route_body(a, smem, true);
}

// Multi-CTA path, step 1: top-k + gates for kChunkTokens tokens per CTA
// (one warp per token, all of the chunk's tokens at once), and the CTA's
// expert histogram.
constexpr int kTopkThreads = kChunkTokens * 32;
__global__ void __launch_bounds__(kTopkThreads) topk_chunk_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                         int32_t *idx, float *gates, int32_t *chunk_counts) {
  __shared__ int s_count[kMaxExperts];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int i = tid; i < E; i += blockDim.x) s_count[i] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kChunkTokens, t1 = min(T, t0 + kChunkTokens);
  for (int t = t0 + w; t < t1; t += blockDim.x >> 5) {
    const int e = warp_topk_softmax(logits + (size_t)t * E, E, k, idx + (size_t)t * k, gates + (size_t)t * k);
    if (lane < k) atomicAdd(&s_count[e], 1);
  }
  __syncthreads();
  if (chunk_counts)
    for (int i = tid; i < E; i += blockDim.x) chunk_counts[(size_t)blockIdx.x * E + i] = s_count[i];
}

// Histogram of given expert ids per chunk (stateless permute).
__global__ void __launch_bounds__(256) hist_chunk_kernel(const int32_t *__restrict__ idx, int T, int k, int E,
                                                         int32_t *chunk_counts) {
  __shared__ int s_count[kMaxExperts];
  const int tid = threadIdx.x;
  for (int i = tid; i < E; i += blockDim.x) s_count[i] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kChunkTokens * k, p1 = min(T, (blockIdx.x + 1) * kChunkTokens) * k;
  for (int p = p0 + tid; p < p1; p += blockDim.x) {
    const int e = idx[p];
    if (e >= 0 && e < E) atomicAdd(&s_count[e], 1);   // out-of-range ids are not counted
  }
  __syncthreads();
  for (int i = tid; i < E; i += blockDim.x) chunk_counts[(size_t)blockIdx.x * E + i] = s_count[i];
}

// Multi-CTA path, step 2 (one CTA): per-expert totals and offsets, each
// chunk's starting position per expert, then (with_plan) the cache plan.
__global__ void __launch_bounds__(kRouteThreads) plan_kernel(RouteArgs a, int with_plan) {
  extern __shared__ int smem[];
  const int E = a.E;
  int *s_count = smem;
  int *s_uexp = s_count + E;
  int *s_victim = s_uexp + E;
  int *s_off = s_victim + E;
  int *s_warp = s_off + E;             // 33
  unsigned *s_bits = (unsigned *)(s_warp + 33);
  int *s_part = (int *)(s_bits + ((a.S + 31) >> 5));   // [G][E]
  const int tid = threadIdx.x;
  // G groups of threads per expert, each summing a contiguous range of chunks
  const int G = max(1, (int)blockDim.x / E);
  const int e = tid % E, g = tid / E;
  const int per = (a.n_chunks + G - 1) / G;
  const int c0 = min(a.n_chunks, g * per), c1 = min(a.n_chunks, c0 + per);
  if (g < G) {
    int part = 0;
    for (int c = c0; c < c1; ++c) part += a.chunk_counts[(size_t)c * E + e];
    s_part[g * E + e] = part;
  }
  __syncthreads();
  int cnt = 0;
  if (tid < E)
    for (int gg = 0; gg < G; ++gg) {   // exclusive prefix over the groups, per expert
      const int p = s_part[gg * E + tid];
      s_part[gg * E + tid] = cnt;
      cnt += p;
    }
  int total;
  const int off = block_excl_scan(tid < E ? cnt : 0, s_warp, &total);
  if (tid < E) {
    s_count[tid] = cnt;
    a.plan.offsets[tid] = off;
    s_off[tid] = off;
  }
  if (tid == 0) a.plan.offsets[E] = total;
  __syncthreads();
  if (g < G) {
    int run = s_off[e] + s_part[g * E + e];
    for (int c = c0; c < c1; ++c) {
      a.chunk_base[(size_t)c * E + e] = run;
      run += a.chunk_counts[(size_t)c * E + e];
    }
  }
  __syncthreads();
  if (with_plan) {
    PlanSmem sm{s_count, s_uexp, s_victim, s_bits, s_warp, nullptr, nullptr, s_off};
    Prefetch pf;
    pf.n = -1;
    if (tid == 0)
      for (int i = 0; i < 5; ++i) pf.st[i] = a.cache.stats[i];
    block_plan(a, sm, pf);
  }
}

// Multi-CTA path, step 3: stable scatter of each chunk's pairs.
__global__ void __launch_bounds__(256) scatter_chunk_kernel(const int32_t *__restrict__ idx, int T, int k, int E,
                                                            const int32_t *__restrict__ chunk_base, int32_t *perm,
                                                            int32_t *inv) {
  extern __shared__ int smem[];
  int *s_base = smem;         // E
  int *s_wcnt = smem + E;     // 8*E
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_base[i] = chunk_base[(size_t)blockIdx.x * E + i];
  __syncthreads();
  const int p0 = blockIdx.x * kChunkTokens * k, p1 = min(T, (blockIdx.x + 1) * kChunkTokens) * k;
  block_rank_scatter(idx, p0, p1, E, s_base, s_wcnt, perm, inv);
}

// Threads of the single-CTA routing kernel: at least E (one per expert in
// the plan), at least 256, enough that each thread's share of the recency
// list (S slots) fits the kPre entries it loads before the wait on the
// kernel ahead (S = 6144 slots: 768 threads), a whole number of warps.
int small_threads(int E, int S) {
  const int for_slots = (S + kPre - 1) / kPre;
  return std::min(kRouteThreads, std::max({256, (E + 31) / 32 * 32, (for_slots + 31) / 32 * 32}));
}

// Both single-CTA bodies: 6 E-sized arrays, 33 scan partials, the general
// path's per-warp counts (nw*E) or the decode path's 68 pair and plan ints,
// and the hit bitmap.
size_t small_smem_bytes(int E, int S) {
  const size_t nw = small_threads(E, S) / 32;
  return sizeof(int) * (6 * (size_t)E + 33 + std::max<size_t>(nw * (size_t)E, 68)) +
         sizeof(unsigned) * (((size_t)S + 31) / 32);
}
size_t plan_smem_bytes(int E, int S) {
  return sizeof(int) * (4 * (size_t)E + 33) + sizeof(unsigned) * (((size_t)S + 31) / 32) +
         sizeof(int) * (size_t)kRouteThreads;   // per-group chunk partials
}

}  // namespace

size_t route_small_smem(int E, int S) { return small_smem_bytes(E, S); }

void route_init_attributes() {
  cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(scatter_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
}

static int n_chunks_of(int T) { return (T + kChunkTokens - 1) / kChunkTokens; }

size_t permute_scratch_ints(int T, int k, int E) {
  (void)k;
  return 2 * (size_t)n_chunks_of(T) * (size_t)E;
}

int route_kernel_count(int T, int k) { return T * k <= kSmallRoutePairs ? 1 : 3; }

// Small calls (T*k <= kSmallRoutePairs) route in one CTA; larger ones in
// three kernels over kChunkTokens-token chunks.
cudaError_t launch_route(const RouteArgs &a, cudaStream_t s) {
  if (a.T * a.k <= kSmallRoutePairs || a.chunk_counts == nullptr) {
    return launch_k(route_small_kernel, dim3(1), dim3(small_threads(a.E, a.S)), small_smem_bytes(a.E, a.S), s,
                    a.pdl != 0, a);
  }
  RouteArgs b = a;
  b.n_chunks = n_chunks_of(a.T);
  topk_chunk_kernel<<<b.n_chunks, kTopkThreads, 0, s>>>(a.logits, a.T, a.E, a.k, a.plan.topk_idx, a.plan.gates,
                                               b.chunk_counts);
  plan_kernel<<<1, kRouteThreads, plan_smem_bytes(a.E, a.S), s>>>(b, 1);
  scatter_chunk_kernel<<<b.n_chunks, 256, sizeof(int) * 9 * (size_t)a.E, s>>>(
      a.plan.topk_idx, a.T, a.k, a.E, b.chunk_base, a.plan.perm, a.plan.inv);
  return cudaGetLastError();
}

cudaError_t launch_topk_only(const float *logits, int T, int E, int k, int32_t *idx, float *gates,
                             cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  topk_chunk_kernel<<<n_chunks_of(T), kTopkThreads, 0, s>>>(logits, T, E, k, idx, gates, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_permute_only(const int32_t *idx, int T, int k, int E, int32_t *offsets, int32_t *perm,
                                int32_t *inv, int32_t *chunk_counts, int32_t *chunk_base, cudaStream_t s) {
  RouteArgs a{};
  a.T = T; a.k = k; a.E = E; a.S = 1;
  a.plan.offsets = offsets;
  a.chunk_counts = chunk_counts;
  a.chunk_base = chunk_base;
  a.n_chunks = n_chunks_of(T);
  if (T > 0) hist_chunk_kernel<<<a.n_chunks, 256, 0, s>>>(idx, T, k, E, chunk_counts);
  plan_kernel<<<1, kRouteThreads, plan_smem_bytes(E, 1), s>>>(a, 0);
  if (T > 0)
    scatter_chunk_kernel<<<a.n_chunks, 256, sizeof(int) * 9 * (size_t)E, s>>>(idx, T, k, E, chunk_base, perm, inv);
  return cudaGetLastError();
}

}  // namespace ftmoe
