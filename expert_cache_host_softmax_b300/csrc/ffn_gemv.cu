// ffn_gemv.cu -- grouped SwiGLU expert FFN for small token groups (decode),
// with the weight dequantisation fused into the dot products, and the
// gate-weighted combine.
//
// Per distinct expert u of a call (its blob sits in slot u_slot[u]) and its
// group of tokens (permuted positions offsets[e] .. offsets[e+1]):
//   gate/up:  h[p][r] = bf16( silu(g) * u ),  g = W_g[r] . x_t,  u = W_u[r] . x_t
//   down:     y[p][n] = W_d[n] . h[p]                       (fp32)
//   combine:  out[t][n] = sum_j gates[t][j] * y[inv[t*k+j]][n], j ascending
// Decode (1..4 tokens per expert) reads each weight once per call and does
// 1..4 multiply-adds with it: bound by HBM bytes and by latency, not by the
// contraction, so this path uses CUDA cores.  What matters is bytes in
// flight and the length of each CTA's chain of dependent loads: 8-32 lanes
// share one weight row, every lane issues its 16-byte loads for a batch of
// chunks before it computes, a CTA reads its plan entry in one 16-byte load,
// and the grid has one CTA per 8-16 output features per expert.  Activations
// are staged once per CTA in shared memory.  With FT_MISS_KERNEL the gate/up
// grid's first rows are copying CTAs (see copy_misses).
//
// For small calls the combine is fused into the down projection: each CTA
// counts itself done on a per-feature-tile counter, and the last CTA of a tile
// sums that tile's outputs over the call's tokens (in rank order) and resets
// the counter for the next call.
//
// Formats: NVFP4 (e2m1 codes, E4M3 scale per 16, fp32 global scale per
// matrix), MXFP4 (e2m1 codes, E8M0 scale per 32; OCP Microscaling v1.0),
// FP8 (E4M3 codes, fp32 scale per row, applied to the finished dot product),
// BF16.  FP4 code bytes hold element 2j in the low nibble.
#include <algorithm>

#include "ft_internal.cuh"

#include "gemv_dev.cuh"

namespace ftmoe {

namespace {

// One CTA: kWarps * 32 / LPR * fpw output features (block blockIdx.x) of one
// distinct expert (blockIdx.y).  With combine counters (down only), the last
// CTA of each feature block also writes that block of the combined output.
// COH (gate/up grids whose own CTAs copy misses into their slots): weights
// are loaded through L2 (ld.global.cg), not through the read-only path, which
// is defined only for data no one writes while the kernel runs.
template <int FMT, bool DOWN, int NT, int LPR, bool COH>
__global__ void __launch_bounds__(kWarps * 32) ffn_gemv_kernel(FfnArgs a, CombineArgs cb, int fpw) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
  // Roles.  Without in-kernel copies, CTA (x, y) works on feature block x of
  // distinct expert y.  With them (copy_rows > 0), roles go by arrival, not by
  // block index (CUDA does not promise an order of dispatch): when the call
  // has misses, the first copy_rows * gridDim.x CTAs to take a ticket copy,
  // and the others take the work items in ticket order, hits first, so the
  // copiers are running before any CTA waits for them, whatever the order of
  // dispatch; when it has none, the first tickets take the work items and the
  // last copy_rows * gridDim.x CTAs have nothing to do.  The ticket counter
  // was last used by the gate/up grid two kernels back, which has completed;
  // the CTA that takes the last ticket re-arms it.
  int item_y = blockIdx.y, item_x = blockIdx.x;
  long long copier = -1;
  int ticket = -1;
  if constexpr (!DOWN) {
    if (a.copy_rows > 0) {
      __shared__ int s_ticket;
      if (threadIdx.x == 0) {
        const int total = gridDim.x * gridDim.y;
        const int t = atomicAdd(a.copy_sync + 2, 1);
        if (t == total - 1) a.copy_sync[2] = 0;
        s_ticket = t;
      }
      __syncthreads();
      ticket = s_ticket;
    }
  }
  // Before the wait for the kernel ahead: this grid starts only once that
  // kernel is past its own wait (it triggers after it), so all work before
  // the route kernel -- the call's x -- and the route kernel's plan (for a
  // down grid, which starts after the gate/up grid passed its wait) are final.
  bool x_staged = false;
  if constexpr (!DOWN) {
    if (NT == 1 && a.max_tokens == 1) {
      // one-token call: every expert multiplies the same row
      stage_row1<FMT, false>(xs, a.x, a.H);
      __syncthreads();
      x_staged = true;
    }
  } else {
    gemv_prefetch<FMT, true, LPR, kWarps>(a, blockIdx.y, blockIdx.x, fpw, false);
  }
  pdl_wait();      // the plan, activations and slots come from earlier kernels
  pdl_trigger();
  if constexpr (!DOWN) {
    if (ticket >= 0) {
      const int nct = a.copy_rows * gridDim.x;
      if (__ldcg(a.mc.n + 2) > 0) {
        if (ticket < nct) {
          copier = ticket;
        } else {
          item_y = a.copy_rows + (ticket - nct) / gridDim.x;
          item_x = (ticket - nct) % gridDim.x;
        }
      } else {
        // no misses: the items take the first tickets, the last nct CTAs exit
        const int items = ((int)gridDim.y - a.copy_rows) * gridDim.x;
        if (ticket >= items) return;
        item_y = a.copy_rows + ticket / gridDim.x;
        item_x = ticket % gridDim.x;
      }
    }
  }
  if constexpr (!DOWN) {
    if (copier >= 0) {
      // a copying CTA: gate/up bytes of every miss, the flag, then the down bytes
      const long long nct = (long long)a.copy_rows * gridDim.x;
      const long long t = copier * blockDim.x + threadIdx.x;
      copy_misses(a.mc, 0, 2, t, nct * blockDim.x);
      cta_arrive_last_sets(a.copy_sync + 1, a.copy_sync, (int)nct, a.seq_raised);
      copy_misses(a.mc, 2, 3, t, nct * blockDim.x);
      return;
    }
  }
  gemv_block<FMT, DOWN, NT, LPR, kWarps, COH>(a, item_y - (DOWN ? 0 : a.copy_rows), item_x, fpw, xs, x_staged);
  if constexpr (DOWN) {
    if (cb.counters == nullptr) return;
    __shared__ int s_last;
    combine_block(a, cb, blockIdx.x, kWarps * (32 / LPR) * fpw, gridDim.y * max(1, cb.launches), &s_last);
  }
}

__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ y, const float *__restrict__ gates,
                                                      const int32_t *__restrict__ inv, int k, int H,
                                                      __nv_bfloat16 *__restrict__ out) {
  const int t = blockIdx.y;
  const int n4 = blockIdx.x * blockDim.x + threadIdx.x;  // index of 4 features
  if (n4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const float g = gates[(size_t)t * k + j];
    const float4 v = __ldg(reinterpret_cast<const float4 *>(y + (size_t)inv[(size_t)t * k + j] * H) + n4);
    acc.x = fmaf(g, v.x, acc.x);
    acc.y = fmaf(g, v.y, acc.y);
    acc.z = fmaf(g, v.z, acc.z);
    acc.w = fmaf(g, v.w, acc.w);
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t *>(&lo);
  pk.y = *reinterpret_cast<uint32_t *>(&hi);
  reinterpret_cast<uint2 *>(out + (size_t)t * H)[n4] = pk;
}

// Lanes per weight row: a power of two dividing the row's 32-element chunks,
// as large as leaves each lane >= 8 chunks for rows shorter than 4096 (>= 4
// for longer rows, whose CTAs already take 4 features a warp; fewer lanes per
// row for short rows).  Eight chunks a lane halves the CTA count against
// four: a decode gate/up grid over 8 experts of H = 2048, I = 768 is then 384
// work CTAs, one wave at 5 CTAs per SM, where 768 left a second wave of 28.
int lanes_per_row(int K) {
  const int chunks = K / 32;
  const int min_per_lane = K >= 4096 ? 4 : 8;
  for (int l : {32, 16, 8})
    if (chunks % l == 0 && chunks / l >= min_per_lane) return l;
  for (int l : {32, 16, 8})
    if (chunks % l == 0) return l;
  return 8;
}

template <int FMT, bool DOWN, int NT, int LPR>
cudaError_t launch_t(const FfnArgs &a, const CombineArgs &cb, cudaStream_t s) {
  const int feats = DOWN ? a.H : a.I;
  const int K = DOWN ? a.I : a.H;
  const int fpw = K >= 4096 ? 4 : 1;
  const int fpc = kWarps * (32 / LPR) * fpw;
  dim3 grid((feats + fpc - 1) / fpc, a.umax + (DOWN ? 0 : a.copy_rows));
  const size_t smem = (size_t)NT * K * sizeof(__nv_bfloat16) + 16;   // + the one-token row's scale
  if constexpr (!DOWN)
    if (a.miss_coherent)
      return launch_k(ffn_gemv_kernel<FMT, false, NT, LPR, true>, grid, dim3(kWarps * 32), smem, s, a.pdl != 0, a,
                      cb, fpw);
  return launch_k(ffn_gemv_kernel<FMT, DOWN, NT, LPR, false>, grid, dim3(kWarps * 32), smem, s, a.pdl != 0, a, cb,
                  fpw);
}

template <int FMT, bool DOWN, int NT>
cudaError_t launch_l(const FfnArgs &a, const CombineArgs &cb, cudaStream_t s) {
  const int l = lanes_per_row(DOWN ? a.I : a.H);
  if (l == 32) return launch_t<FMT, DOWN, NT, 32>(a, cb, s);
  if (l == 16) return launch_t<FMT, DOWN, NT, 16>(a, cb, s);
  return launch_t<FMT, DOWN, NT, 8>(a, cb, s);
}

template <int FMT, bool DOWN>
cudaError_t launch_n(const FfnArgs &a, const CombineArgs &cb, cudaStream_t s) {
  // no expert of a call sees more tokens than the call has
  if (a.max_tokens <= 1) return launch_l<FMT, DOWN, 1>(a, cb, s);
  if (a.max_tokens == 2) return launch_l<FMT, DOWN, 2>(a, cb, s);
  return launch_l<FMT, DOWN, 4>(a, cb, s);
}

template <bool DOWN>
cudaError_t launch_ffn(const FfnArgs &a, const CombineArgs &cb, cudaStream_t s) {
  switch (a.fmt) {
    case FMT_BF16: return launch_n<FMT_BF16, DOWN>(a, cb, s);
    case FMT_NVFP4: return launch_n<FMT_NVFP4, DOWN>(a, cb, s);
    case FMT_FP8: return launch_n<FMT_FP8, DOWN>(a, cb, s);
    default: return launch_n<FMT_MXFP4, DOWN>(a, cb, s);
  }
}

template <int FMT, bool DOWN, int NT, bool COH>
void attr_c() {
  const int max_smem = NT * 8192 * 2 + 16;   // activations of NT token rows, K <= 8192
  cudaFuncSetAttribute(ffn_gemv_kernel<FMT, DOWN, NT, 8, COH>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(ffn_gemv_kernel<FMT, DOWN, NT, 16, COH>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(ffn_gemv_kernel<FMT, DOWN, NT, 32, COH>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

template <int FMT, bool DOWN, int NT>
void attr_l() {
  attr_c<FMT, DOWN, NT, false>();
  if constexpr (!DOWN) attr_c<FMT, DOWN, NT, true>();
}

template <int FMT>
void attr_f() {
  attr_l<FMT, false, 1>(); attr_l<FMT, false, 2>(); attr_l<FMT, false, 4>();
  attr_l<FMT, true, 1>(); attr_l<FMT, true, 2>(); attr_l<FMT, true, 4>();
}

}  // namespace

void ffn_init_attributes() {
  attr_f<FMT_BF16>();
  attr_f<FMT_NVFP4>();
  attr_f<FMT_MXFP4>();
  attr_f<FMT_FP8>();
}

int combine_tiles(int H) { return (H + kMinFeatPerCta - 1) / kMinFeatPerCta; }

int gateup_feature_blocks(int H, int I) {
  const int fpc = kWarps * (32 / lanes_per_row(H)) * (H >= 4096 ? 4 : 1);
  return (I + fpc - 1) / fpc;
}

bool gemv_fuses_combine(int T) { return T <= kFusedCombineMaxT; }

cudaError_t launch_gateup(const FfnArgs &a, cudaStream_t s) { return launch_ffn<false>(a, CombineArgs{}, s); }

cudaError_t launch_down(const FfnArgs &a, const CombineArgs &cb, cudaStream_t s) { return launch_ffn<true>(a, cb, s); }

__global__ void __launch_bounds__(256) acc_to_bf16_kernel(const float4 *__restrict__ acc, uint2 *__restrict__ out,
                                                          int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = __ldcs(acc + i);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    out[i] = pk;
  }
}

cudaError_t launch_acc_to_bf16(const float *acc, __nv_bfloat16 *out, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int64_t n4 = n / 4;
  const int grid = (int)std::min<int64_t>((n4 + 255) / 256, 148 * 8);
  acc_to_bf16_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4 *>(acc), reinterpret_cast<uint2 *>(out), n4);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float *y, const float *gates, const int32_t *inv, int T, int k, int H,
                           __nv_bfloat16 *out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dim3 grid((H / 4 + 255) / 256, T);
  combine_kernel<<<grid, 256, 0, s>>>(y, gates, inv, k, H, out);
  return cudaGetLastError();
}

}  // namespace ftmoe
