// decode_layer.cu -- one decode layer call (LRU mode, a few tokens) as a single
// cooperative kernel.
//
// A decode call moves little data: the cost of the path route -> gate/up ->
// down as separate kernels is mostly their launch and ramp latencies.  Here
// one grid, all of whose CTAs are resident (cooperative launch), runs:
//   A. CTA 0: top-k + softmax, permute and the LRU plan (the routing kernel's
//      code); it publishes the miss list to the host and raises a plan flag.
//      The other CTAs wait for the flag (bounded).
//   B. gate/up GEMV of the hits (all CTAs, work items (expert, feature block)).
//   C. if the call has misses: wait until the copy stream has landed them (a
//      4-byte flag the copy stream writes after the expert copies, bounded),
//      then gate/up of the misses.  With FT_MISS_PULL the misses are read over
//      PCIe in B instead, and C has nothing to do.
//   D. grid barrier (bounded).
//   E. down GEMV of all experts, with the combine fused in (the last CTA of
//      each feature block sums it over the call's tokens).
// The per-call hit/miss/copy semantics are those of the multi-kernel path
// ("Why a Huge MoE Model Fits on One Consumer GPU": a cached expert runs at
// GPU speed, a miss is streamed over PCIe, and the hits' work overlaps the
// copies).
#include "gemv_dev.cuh"
#include "route_dev.cuh"
#include "wait_dev.cuh"

namespace ftmoe {

namespace {

constexpr int kMegaWarps = 8;
constexpr int kMegaThreads = kMegaWarps * 32;
// Grid-wide barrier over G resident CTAs (bounded).  count returns to 0 after
// each use; gen only grows.
__device__ __forceinline__ bool grid_barrier(int *count, int *gen, int G, int *err, int site, int *s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const volatile int *vg = gen;
    const int g = *vg;
    bool ok = true;
    __threadfence();
    if (atomicAdd(count, 1) == G - 1) {
      atomicExch(count, 0);
      __threadfence();
      atomicAdd(gen, 1);
    } else {
      const unsigned long long t0 = dev_timer_ns();
      while (*vg == g) {
        if (dev_timer_ns() - t0 > kWaitNs) {
          atomicCAS(err, 0, site);
          ok = false;
          break;
        }
      }
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

struct MegaArgs {
  RouteArgs r;        // routing and plan; r.mirror = host mirror (null with FT_MISS_PULL)
  FfnArgs f;
  CombineArgs cb;     // combine counters: one per down feature block
  int *sync;          // [0] plan flag, [1] copy flag (written by the copy stream), [2] barrier count, [3] generation
  int lpr_gu, lpr_dn, fpw_gu, fpw_dn;
  int nb_gu, nb_dn;   // feature blocks per expert
  int wait_copies;    // misses arrive by copy: wait for the copy flag before their gate/up
};

// Every load of weights and h goes through L2 (coherent): the misses' slots
// are written while the kernel runs (by the copy engine, or by its own CTAs
// pulling them from host memory), and so is h.
template <int FMT, bool DOWN, int NT>
__device__ __forceinline__ void gemv_item(const FfnArgs &a, int lpr, int u, int bx, int fpw, __nv_bfloat16 *xs) {
  if (lpr == 32) gemv_block<FMT, DOWN, NT, 32, kMegaWarps, true>(a, u, bx, fpw, xs);
  else if (lpr == 16) gemv_block<FMT, DOWN, NT, 16, kMegaWarps, true>(a, u, bx, fpw, xs);
  else gemv_block<FMT, DOWN, NT, 8, kMegaWarps, true>(a, u, bx, fpw, xs);
}

template <int FMT, bool DOWN>
__device__ __forceinline__ void prefetch_item(const FfnArgs &a, int lpr, int u, int bx, int fpw, bool any) {
  if (lpr == 32) gemv_prefetch<FMT, DOWN, 32, kMegaWarps>(a, u, bx, fpw, any);
  else if (lpr == 16) gemv_prefetch<FMT, DOWN, 16, kMegaWarps>(a, u, bx, fpw, any);
  else gemv_prefetch<FMT, DOWN, 8, kMegaWarps>(a, u, bx, fpw, any);
}

template <int FMT, int NT>
__global__ void __launch_bounds__(kMegaThreads) decode_layer_kernel(MegaArgs m) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_ok, s_last;
  __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
  const int G = gridDim.x;
  const uint32_t seq = m.r.seq;
  int *err = m.f.err;

  // ---- A. routing and plan (CTA 0)
  if (blockIdx.x == 0) {
    route_body(m.r, reinterpret_cast<int *>(smem_raw), false);
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      atomicExch(m.sync, (int)seq);
    }
  }
  if (!cta_wait_flag(m.sync, (int)seq, err, 60, &s_ok)) return;
  const int n_u = __ldcg(m.r.plan.n), n_miss = __ldcg(m.r.plan.n + 2);

  // ---- B. gate/up of the hits (or of every expert when misses are pulled);
  // this CTA's hit weight rows are requested from L2 first, all at once
  FfnArgs fa = m.f;
  fa.only = m.wait_copies ? 1 : 0;
  for (int it = blockIdx.x; it < n_u * m.nb_gu; it += G)
    prefetch_item<FMT, false>(fa, m.lpr_gu, it / m.nb_gu, it % m.nb_gu, m.fpw_gu, false);
  for (int it = blockIdx.x; it < n_u * m.nb_gu; it += G)
    gemv_item<FMT, false, NT>(fa, m.lpr_gu, it / m.nb_gu, it % m.nb_gu, m.fpw_gu, xs);

  // ---- C. gate/up of the misses, once the copy stream has landed them
  if (m.wait_copies && n_miss > 0) {
    if (!cta_wait_flag(m.sync + 1, (int)seq, err, 61, &s_ok)) return;
    fa.only = 2;
    for (int it = blockIdx.x; it < n_u * m.nb_gu; it += G)
      gemv_item<FMT, false, NT>(fa, m.lpr_gu, it / m.nb_gu, it % m.nb_gu, m.fpw_gu, xs);
  }

  // ---- D. every h row is written; the down rows are requested meanwhile
  for (int it = blockIdx.x; it < n_u * m.nb_dn; it += G)
    prefetch_item<FMT, true>(fa, m.lpr_dn, it / m.nb_dn, it % m.nb_dn, m.fpw_dn, true);
  if (!grid_barrier(m.sync + 2, m.sync + 3, G, err, 62, &s_ok)) return;

  // ---- E. down, with the combine fused per feature block
  fa.only = 0;
  const int feat_per_block = kMegaWarps * (32 / m.lpr_dn) * m.fpw_dn;
  for (int it = blockIdx.x; it < n_u * m.nb_dn; it += G) {
    const int u = it / m.nb_dn, bx = it % m.nb_dn;
    gemv_item<FMT, true, NT>(fa, m.lpr_dn, u, bx, m.fpw_dn, xs);
    combine_block(fa, m.cb, bx, feat_per_block, n_u, &s_last);
  }
}

template <int FMT, int NT>
cudaError_t launch_mega(const MegaArgs &m, int grid, size_t smem, cudaStream_t s) {
  void *args[] = {const_cast<MegaArgs *>(&m)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(decode_layer_kernel<FMT, NT>), dim3(grid),
                                     dim3(kMegaThreads), args, smem, s);
}

template <int FMT, int NT>
int mega_capacity(size_t smem) {
  int dev = 0, sms = 0, per = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaFuncSetAttribute(decode_layer_kernel<FMT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, decode_layer_kernel<FMT, NT>, kMegaThreads, smem) !=
      cudaSuccess)
    return 0;
  return per * sms;
}

int lanes_per_row_m(int K) {
  const int chunks = K / 32;
  for (int l : {32, 16, 8})
    if (chunks % l == 0 && chunks / l >= 4) return l;
  for (int l : {32, 16, 8})
    if (chunks % l == 0) return l;
  return 8;
}

}  // namespace

bool mega_supported(int E, int T, int k) { return E <= kMegaThreads && T * k <= kSmallRoutePairs && T <= 16; }

int mega_counters(int H) { return (H + kMegaWarps - 1) / kMegaWarps; }

// One decode layer call.  `route`, `ffn` and `cb` are filled as for the
// multi-kernel path; sync: 4 device ints (zero at create and reset).
// route_smem: shared memory of the routing code.
cudaError_t launch_decode_layer(const RouteArgs &route, const FfnArgs &ffn, const CombineArgs &cb, int *sync,
                                bool wait_copies, size_t route_smem, cudaStream_t s) {
  MegaArgs m{};
  m.r = route;
  m.f = ffn;
  m.cb = cb;
  m.sync = sync;
  m.wait_copies = wait_copies ? 1 : 0;

  m.lpr_gu = lanes_per_row_m(ffn.H);
  m.lpr_dn = lanes_per_row_m(ffn.I);
  m.fpw_gu = ffn.H >= 4096 ? 4 : 1;
  m.fpw_dn = ffn.I >= 4096 ? 4 : 1;
  m.nb_gu = ffn.I / (kMegaWarps * (32 / m.lpr_gu) * m.fpw_gu);
  m.nb_dn = ffn.H / (kMegaWarps * (32 / m.lpr_dn) * m.fpw_dn);
  const int NT = ffn.max_tokens <= 1 ? 1 : ffn.max_tokens == 2 ? 2 : 4;
  const size_t smem = std::max(route_smem, (size_t)NT * std::max(ffn.H, ffn.I) * 2 + 16);
  // resident CTAs per launch configuration (cached: the query costs host time)
  static int cap[3][3] = {};
  static size_t cap_smem[3][3] = {};
  if (ffn.fmt < FMT_BF16 || ffn.fmt > FMT_MXFP4) return cudaErrorInvalidValue;   // BF16, NVFP4, MXFP4 only
  const int fi = ffn.fmt, ni = NT == 1 ? 0 : NT == 2 ? 1 : 2;
  if (cap[fi][ni] == 0 || cap_smem[fi][ni] != smem) {
    cap_smem[fi][ni] = smem;
    switch (fi * 3 + ni) {
      case 0: cap[fi][ni] = mega_capacity<FMT_BF16, 1>(smem); break;
      case 1: cap[fi][ni] = mega_capacity<FMT_BF16, 2>(smem); break;
      case 2: cap[fi][ni] = mega_capacity<FMT_BF16, 4>(smem); break;
      case 3: cap[fi][ni] = mega_capacity<FMT_NVFP4, 1>(smem); break;
      case 4: cap[fi][ni] = mega_capacity<FMT_NVFP4, 2>(smem); break;
      case 5: cap[fi][ni] = mega_capacity<FMT_NVFP4, 4>(smem); break;
      case 6: cap[fi][ni] = mega_capacity<FMT_MXFP4, 1>(smem); break;
      case 7: cap[fi][ni] = mega_capacity<FMT_MXFP4, 2>(smem); break;
      default: cap[fi][ni] = mega_capacity<FMT_MXFP4, 4>(smem); break;
    }
  }
  const int items = ffn.umax * std::max(m.nb_gu, m.nb_dn);
  const int grid = std::max(1, std::min(cap[fi][ni], items));
  if (cap[fi][ni] <= 0) return cudaErrorCooperativeLaunchTooLarge;
  switch (fi * 3 + ni) {
    case 0: return launch_mega<FMT_BF16, 1>(m, grid, smem, s);
    case 1: return launch_mega<FMT_BF16, 2>(m, grid, smem, s);
    case 2: return launch_mega<FMT_BF16, 4>(m, grid, smem, s);
    case 3: return launch_mega<FMT_NVFP4, 1>(m, grid, smem, s);
    case 4: return launch_mega<FMT_NVFP4, 2>(m, grid, smem, s);
    case 5: return launch_mega<FMT_NVFP4, 4>(m, grid, smem, s);
    case 6: return launch_mega<FMT_MXFP4, 1>(m, grid, smem, s);
    case 7: return launch_mega<FMT_MXFP4, 2>(m, grid, smem, s);
    default: return launch_mega<FMT_MXFP4, 4>(m, grid, smem, s);
  }
}

}  // namespace ftmoe
