// decode_grid.cu -- one decode call (LRU mode, GEMV, misses copied on the
// GPU, at most 32 (token, rank) pairs) as a single grid.
//
// "FreeToken: Run Frontier MoE Models on Your Own GPU, and the RAM It Takes",
// section "Why a Huge MoE Model Fits on One Consumer GPU": a cached expert
// runs at GPU speed; a miss is streamed over PCIe.  The work of the call --
// route and plan, the misses' copies from pinned host memory, the gate/up
// GEMV of every distinct expert, the down GEMV and the combine -- is one grid
// whose CTAs take their role by arrival ticket, not by block index (CUDA
// promises no order of dispatch):
//   ticket 0                 the router: top-k + softmax, permute and the LRU
//                            plan (the routing kernel's decode body), then the
//                            plan flag;
//   the next C tickets       copiers: gate/up bytes of every miss, flag A, then
//                            the down bytes, flag B;
//   the next U * NB_gu       gate/up items (distinct expert u in plan order,
//                            hits first; feature block bx); a miss's items wait
//                            for flag A; each item counts itself done per u;
//   the last U * NB_dn       down items; wait until expert u's gate/up items are
//                            all done (and for a miss, flag B); the combine of a
//                            feature block is done by its last item.
// Every wait is on CTAs with smaller tickets, which are already running, so
// the grid makes progress whatever the order of dispatch; every wait is
// bounded (kWaitNs, then an error code in the device word).  The hits' FFN
// runs while the copiers stream the misses.  Flags carry the call's sequence
// number, so a flag left from an earlier call never matches.
//
// Programmatic dependent launch: a CTA lets the next call's grid launch only
// once it has seen this call's plan flag, so the router of the next call (which
// reads the cache tables before it waits for this grid to complete) finds the
// tables final, and the next grid's CTAs are dispatched only after all of this
// grid's.  Loads of slot bytes and of h go through L2 (ld.global.cg): misses'
// slots and h are written while the grid runs.
#include <algorithm>

#include "gemv_dev.cuh"
#include "route_dev.cuh"
#include "wait_dev.cuh"

namespace ftmoe {

namespace {

constexpr int kGridThreads = kWarps * 32;

struct GridArgs {
  RouteArgs r;
  FfnArgs f;              // f.mc: the miss copies; f.copy_rows = 0 (the waits are here)
  CombineArgs cb;
  int *sync;              // see DecodeSync
  int n_copy;             // copier CTAs
  int nb_gu, nb_dn;       // feature blocks per distinct expert
  int lpr_gu, lpr_dn, fpw_gu, fpw_dn;
  int seq, seq_raised;    // the call's sequence number; the value the copiers raise
};

// sync words: [0] plan flag, [1] flag A, [2] count A, [3] flag B, [4] count B,
// [5..6] ticket counters (by call parity), [8 + u] gate/up items done of u.
enum { kPlanFlag = 0, kFlagA = 1, kCountA = 2, kFlagB = 3, kCountB = 4, kTicket = 5, kDone = 8 };

// Bounded wait of thread 0 until *flag == want; the CTA learns the outcome.
// Waiters back off kGridPollNs between polls: hundreds of CTAs may wait on
// one flag, and their polls share one L2 line with the CTA that will raise it.
constexpr unsigned kGridPollNs = 400;
__device__ __forceinline__ bool grid_wait(const int *flag, int want, int *err, int site, int *s_ok) {
  if (threadIdx.x == 0) {
    const volatile int *vf = flag;
    bool ok = true;
    if (*vf != want) {
      const unsigned long long t0 = dev_timer_ns();
      while (*vf != want) {
        if (dev_timer_ns() - t0 > kWaitNs) {
          atomicCAS(err, 0, site);
          ok = false;
          break;
        }
        __nanosleep(kGridPollNs);
      }
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

template <int FMT, bool DOWN, int NT>
__device__ __forceinline__ void grid_gemv(const FfnArgs &a, int lpr, int u, int bx, int fpw, __nv_bfloat16 *xs,
                                          bool x_staged) {
  if (lpr == 32) gemv_block<FMT, DOWN, NT, 32, kWarps, true>(a, u, bx, fpw, xs, x_staged);
  else if (lpr == 16) gemv_block<FMT, DOWN, NT, 16, kWarps, true>(a, u, bx, fpw, xs, x_staged);
  else gemv_block<FMT, DOWN, NT, 8, kWarps, true>(a, u, bx, fpw, xs, x_staged);
}

template <int FMT, int NT>
__global__ void __launch_bounds__(kGridThreads) decode_grid_kernel(GridArgs g) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_ticket, s_ok;
  int *sync = g.sync;
  if (threadIdx.x == 0) {
    const int total = gridDim.x;
    const int t = atomicAdd(sync + kTicket + (g.seq & 1), 1);
    if (t == total - 1) {
      sync[kTicket + (g.seq & 1)] = 0;   // every CTA of this call has its ticket: re-arm
      __threadfence();
    }
    s_ticket = t;
  }
  __syncthreads();
  const int t = s_ticket;
  const int n_gu = g.f.umax * g.nb_gu;

  if (t == 0) {
    // ================================================================ router
    route_decode_body(g.r, reinterpret_cast<int *>(smem_raw), true);   // waits for the previous grid
    if (threadIdx.x < 32) {
      // warp 0 wrote the plan; the recency list was written before its last block barrier
      for (int u = threadIdx.x; u < g.f.umax; u += 32) sync[kDone + u] = 0;
      __threadfence();
      __syncwarp();
      if (threadIdx.x == 0) atomicExch(sync + kPlanFlag, g.seq);
    }
    return;
  }
  // one-token call: every gate/up item multiplies the same x row (the call's
  // input, written before the previous grid; see the header)
  __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
  const bool gu_item = t >= 1 + g.n_copy && t < 1 + g.n_copy + n_gu;
  bool x_staged = false;
  if (NT == 1 && gu_item && g.f.max_tokens == 1) {
    stage_row1<FMT, false>(xs, g.f.x, g.f.H);
    x_staged = true;
  }
  if (!grid_wait(sync + kPlanFlag, g.seq, g.f.err, 80, &s_ok)) return;
  pdl_trigger();   // this call's plan (and the cache tables) are final
  const int nU = __ldcg(g.r.plan.n), n_miss = __ldcg(g.r.plan.n + 2);

  if (t < 1 + g.n_copy) {
    // ================================================================ copier
    if (n_miss == 0) return;
    const long long nct = (long long)g.n_copy * blockDim.x, tt = (long long)(t - 1) * blockDim.x + threadIdx.x;
    copy_misses(g.f.mc, 0, 2, tt, nct);
    cta_arrive_last_sets(sync + kCountA, sync + kFlagA, g.n_copy, g.seq_raised);
    copy_misses(g.f.mc, 2, 3, tt, nct);
    cta_arrive_last_sets(sync + kCountB, sync + kFlagB, g.n_copy, g.seq_raised);
    return;
  }
  if (gu_item) {
    // ================================================================ gate/up
    const int i = t - 1 - g.n_copy, u = i / g.nb_gu, bx = i - u * g.nb_gu;
    if (u >= nU) return;
    const bool hit = __ldcg(&g.r.plan.u_info[u].w) & 1;
    if (!hit && !grid_wait(sync + kFlagA, g.seq, g.f.err, 81, &s_ok)) return;
    grid_gemv<FMT, false, NT>(g.f, g.lpr_gu, u, bx, g.fpw_gu, xs, x_staged);
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(sync + kDone + u, 1);
    }
    return;
  }
  // ================================================================ down (+ combine)
  const int i = t - 1 - g.n_copy - n_gu, u = i / g.nb_dn, bx = i - u * g.nb_dn;
  if (u < nU) {
    bool ok = true;
    if (threadIdx.x == 0) {
      // every gate/up item of u has stored its part of h (bounded wait)
      const volatile int *vd = sync + kDone + u;
      if (*vd != g.nb_gu) {
        const unsigned long long t0 = dev_timer_ns();
        while (*vd != g.nb_gu) {
          if (dev_timer_ns() - t0 > kWaitNs) {
            atomicCAS(g.f.err, 0, 82);
            ok = false;
            break;
          }
          __nanosleep(kGridPollNs);
        }
      }
      __threadfence();
      s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) return;
    const bool hit = __ldcg(&g.r.plan.u_info[u].w) & 1;
    if (!hit && !grid_wait(sync + kFlagB, g.seq, g.f.err, 83, &s_ok)) return;
    grid_gemv<FMT, true, NT>(g.f, g.lpr_dn, u, bx, g.fpw_dn, xs, false);
  }
  __shared__ int s_last;
  combine_block(g.f, g.cb, bx, kWarps * (32 / g.lpr_dn) * g.fpw_dn, g.f.umax, &s_last);
}

int lanes_per_row_g(int K) {
  const int chunks = K / 32;
  for (int l : {32, 16, 8})
    if (chunks % l == 0 && chunks / l >= 4) return l;
  for (int l : {32, 16, 8})
    if (chunks % l == 0) return l;
  return 8;
}

template <int FMT, int NT>
cudaError_t launch_g(const GridArgs &g, int grid, size_t smem, bool pdl, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(decode_grid_kernel<FMT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    attr = true;
  }
  return launch_k(decode_grid_kernel<FMT, NT>, dim3(grid), dim3(kGridThreads), smem, s, pdl, g);
}

template <int FMT>
cudaError_t launch_n(const GridArgs &g, int grid, size_t smem, bool pdl, cudaStream_t s) {
  if (g.f.max_tokens <= 1) return launch_g<FMT, 1>(g, grid, smem, pdl, s);
  if (g.f.max_tokens == 2) return launch_g<FMT, 2>(g, grid, smem, pdl, s);
  return launch_g<FMT, 4>(g, grid, smem, pdl, s);
}

}  // namespace

bool decode_grid_supported(int T, int k, int H, int I) {
  return T * k <= kDecodeRoutePairs && T <= 4 && std::max(H, I) * 2 * 4 <= 96 * 1024;
}

int decode_grid_sync_ints(int umax) { return kDone + umax; }

cudaError_t launch_decode_grid(const RouteArgs &route, const FfnArgs &ffn, const CombineArgs &cb, int *sync,
                               int n_copy, int seq_raised, bool pdl, cudaStream_t s) {
  GridArgs g{};
  g.r = route;
  g.f = ffn;
  g.f.copy_rows = 0;
  g.cb = cb;
  g.sync = sync;
  g.n_copy = n_copy;
  g.lpr_gu = lanes_per_row_g(ffn.H);
  g.lpr_dn = lanes_per_row_g(ffn.I);
  g.fpw_gu = ffn.H >= 4096 ? 4 : 1;
  g.fpw_dn = ffn.I >= 4096 ? 4 : 1;
  const int fpc_gu = kWarps * (32 / g.lpr_gu) * g.fpw_gu, fpc_dn = kWarps * (32 / g.lpr_dn) * g.fpw_dn;
  g.nb_gu = (ffn.I + fpc_gu - 1) / fpc_gu;
  g.nb_dn = (ffn.H + fpc_dn - 1) / fpc_dn;
  g.seq = (int)route.seq;
  g.seq_raised = seq_raised;
  const int NT = ffn.max_tokens <= 1 ? 1 : ffn.max_tokens == 2 ? 2 : 4;
  const size_t route_smem = sizeof(int) * (6 * (size_t)route.E + 33 + 68) + sizeof(unsigned) * (((size_t)route.S + 31) / 32);
  const size_t smem = std::max(route_smem, (size_t)NT * std::max(ffn.H, ffn.I) * 2 + 16);
  if (smem > 96 * 1024) return cudaErrorInvalidValue;
  const int grid = 1 + n_copy + ffn.umax * (g.nb_gu + g.nb_dn);
  switch (ffn.fmt) {
    case FMT_BF16: return launch_n<FMT_BF16>(g, grid, smem, pdl, s);
    case FMT_NVFP4: return launch_n<FMT_NVFP4>(g, grid, smem, pdl, s);
    case FMT_FP8: return launch_n<FMT_FP8>(g, grid, smem, pdl, s);
    default: return launch_n<FMT_MXFP4>(g, grid, smem, pdl, s);
  }
}

}  // namespace ftmoe
