// ffn_gemv.cu -- grouped SwiGLU expert FFN for small token groups (decode),
// with the weight dequantisation fused into the dot products.  Also the
// gate-weighted combine.
//
// Per distinct expert u of a call (its blob sits in slot u_slot[u]) and its
// group of tokens (permuted positions offsets[e] .. offsets[e+1]):
//   gate/up:  h[p][r] = bf16( silu(g) * u ),  g = W_g[r] . x_t,  u = W_u[r] . x_t
//   down:     y[p][n] = W_d[n] . h[p]                       (fp32)
//   combine:  out[t][n] = sum_j gates[t][j] * y[inv[t*k+j]][n], j ascending
// Weight bytes are read once per token chunk of up to 8 tokens.  Decode
// (1..8 tokens per expert) is bound by HBM bytes, not by the contraction, so
// this path uses CUDA cores.  Each warp streams whole weight rows with 16-byte
// loads.  The matching activations are staged once per CTA in shared memory.
//
// Formats: NVFP4 (e2m1 codes, E4M3 scale per 16, fp32 global scale per
// matrix), MXFP4 (e2m1 codes, E8M0 scale per 32; OCP Microscaling v1.0),
// BF16.  Code bytes hold element 2j in the low nibble.
#include "ft_internal.cuh"

namespace ftmoe {

namespace {

constexpr int kFfnThreads = 256;
constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerCta = (kFfnThreads / 32) * kRowsPerWarp;
constexpr int kTokChunk = 8;

// Two e2m1 codes (one byte) -> two halves, via the sm_100-family conversion.
__device__ __forceinline__ __half2 e2m1x2_to_half2(uint32_t byte) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
      : "=r"(out)
      : "r"(byte));
  return *reinterpret_cast<__half2 *>(&out);
}

// Two E4M3 bytes (low byte first) -> two halves.
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint32_t two_bytes) {
  uint32_t out;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(out)
      : "r"(two_bytes));
  return *reinterpret_cast<__half2 *>(&out);
}

// E8M0 scale byte -> 2^(byte-127) (0xFF is NaN).
__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
  if (b == 0xFFu) return __int_as_float(0x7fc00000);
  return __uint_as_float(b ? (b << 23) : 0x00400000u);
}

__device__ __forceinline__ void bf16x8_to_float(const uint4 &v, float *f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Decodes one 32-element chunk c of a weight row into w[32] (without the
// NVFP4 global scale, which is applied to the finished dot product).
template <int FMT>
__device__ __forceinline__ void load_chunk(const uint8_t *__restrict__ codes_row, const uint8_t *__restrict__ sf_row,
                                           int c, float *w) {
  if constexpr (FMT == FMT_BF16) {
    const uint4 *p = reinterpret_cast<const uint4 *>(codes_row) + 4 * c;
#pragma unroll
    for (int i = 0; i < 4; ++i) bf16x8_to_float(__ldg(p + i), w + 8 * i);
  } else {
    const uint4 q = __ldg(reinterpret_cast<const uint4 *>(codes_row) + c);
    float s0, s1;
    if constexpr (FMT == FMT_NVFP4) {
      const uint32_t sb = __ldg(reinterpret_cast<const uint16_t *>(sf_row) + c);
      const float2 s = __half22float2(e4m3x2_to_half2(sb));
      s0 = s.x;
      s1 = s.y;
    } else {
      s0 = s1 = e8m0_to_float(__ldg(sf_row + c));
    }
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 v = __half22float2(e2m1x2_to_half2(words[i] >> (8 * b)));
        const float s = i < 2 ? s0 : s1;  // bytes 0..7 -> elements 0..15 (first block of 16)
        w[8 * i + 2 * b] = v.x * s;
        w[8 * i + 2 * b + 1] = v.y * s;
      }
    }
  }
}

// acc[t] += row . xs[t] over K for NT tokens (lane-partial; caller reduces).
template <int FMT, int NT>
__device__ __forceinline__ void row_dot(const uint8_t *__restrict__ codes_row, const uint8_t *__restrict__ sf_row,
                                        int K, const __nv_bfloat16 *xs, float *acc) {
  const int lane = threadIdx.x & 31;
  for (int c = lane; c < K / 32; c += 32) {
    float w[32];
    load_chunk<FMT>(codes_row, sf_row, c, w);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint4 *xp = reinterpret_cast<const uint4 *>(xs + (size_t)t * K + 32 * c);
      float a = acc[t];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float xf[8];
        bf16x8_to_float(xp[i], xf);
#pragma unroll
        for (int q = 0; q < 8; ++q) a = fmaf(w[8 * i + q], xf[q], a);
      }
      acc[t] = a;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int FMT>
struct RowPtrs {
  const uint8_t *codes, *sf;
};

// Row r of W_gu (r < 2I) or of W_d, inside one blob.
template <int FMT>
__device__ __forceinline__ RowPtrs<FMT> row_ptrs(const uint8_t *blob, const BlobLayout &L, bool down, int r, int K) {
  RowPtrs<FMT> p;
  if constexpr (FMT == FMT_BF16) {
    p.codes = blob + (down ? L.d_codes : L.gu_codes) + (size_t)r * K * 2;
    p.sf = nullptr;
  } else if constexpr (FMT == FMT_NVFP4) {
    p.codes = blob + (down ? L.d_codes : L.gu_codes) + (size_t)r * (K / 2);
    p.sf = blob + (down ? L.d_sf : L.gu_sf) + (size_t)r * (K / 16);
  } else {
    p.codes = blob + (down ? L.d_codes : L.gu_codes) + (size_t)r * (K / 2);
    p.sf = blob + (down ? L.d_sf : L.gu_sf) + (size_t)r * (K / 32);
  }
  return p;
}

template <int FMT, int NT>
__device__ void gateup_rows(const uint8_t *blob, const BlobLayout &L, int H, int I, int row0,
                            const __nv_bfloat16 *xs, int nt, __nv_bfloat16 *h_out /* row p0 of h */,
                            float gs_g, float gs_u) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll 1
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int r = row0 + warp * kRowsPerWarp + rr;
    if (r >= I) break;
    float ag[NT], au[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) ag[t] = au[t] = 0.0f;
    const RowPtrs<FMT> pg = row_ptrs<FMT>(blob, L, false, r, H);
    const RowPtrs<FMT> pu = row_ptrs<FMT>(blob, L, false, I + r, H);
    row_dot<FMT, NT>(pg.codes, pg.sf, H, xs, ag);
    row_dot<FMT, NT>(pu.codes, pu.sf, H, xs, au);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float g = warp_sum(ag[t]) * gs_g;
      const float u = warp_sum(au[t]) * gs_u;
      if (lane == t && t < nt) {
        const float hv = g / (1.0f + expf(-g)) * u;
        h_out[(size_t)t * I + r] = __float2bfloat16_rn(hv);
      }
    }
  }
}

template <int FMT, int NT>
__device__ void down_rows(const uint8_t *blob, const BlobLayout &L, int H, int I, int row0,
                          const __nv_bfloat16 *xs, int nt, float *y_out /* row p0 of y */, float gs_d) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll 1
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int n = row0 + warp * kRowsPerWarp + rr;
    if (n >= H) break;
    float a[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) a[t] = 0.0f;
    const RowPtrs<FMT> pd = row_ptrs<FMT>(blob, L, true, n, I);
    row_dot<FMT, NT>(pd.codes, pd.sf, I, xs, a);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float v = warp_sum(a[t]) * gs_d;
      if (lane == t && t < nt) y_out[(size_t)t * H + n] = v;
    }
  }
}

// One CTA: kRowsPerCta rows of one distinct expert, all of its tokens.
template <int FMT, bool DOWN>
__global__ void __launch_bounds__(kFfnThreads) ffn_gemv_kernel(FfnArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
  const int u = blockIdx.y;
  if (u >= a.plan.n[0]) return;
  const int hit = a.plan.u_hit[u];
  if ((a.only == 1 && !hit) || (a.only == 2 && hit)) return;
  const int e = a.plan.u_expert[u];
  const int off = a.plan.offsets[e];
  const int n = a.plan.offsets[e + 1] - off;
  const uint8_t *blob = a.slot_bank + (size_t)a.plan.u_slot[u] * a.slot_stride;
  const BlobLayout L = blob_layout(FMT, a.H, a.I);
  const int K = DOWN ? a.I : a.H;
  float gs0 = 1.0f, gs1 = 1.0f;
  if constexpr (FMT == FMT_NVFP4) {
    const float *gs = reinterpret_cast<const float *>(blob + L.gscale);
    gs0 = DOWN ? gs[2] : gs[0];
    gs1 = gs[1];
  }
  const int row0 = blockIdx.x * kRowsPerCta;
  for (int c0 = 0; c0 < n; c0 += kTokChunk) {
    const int nt = min(kTokChunk, n - c0);
    // stage the chunk's activations (bf16 rows of K) in shared memory
    const int vec_per_row = K / 8;
    for (int i = threadIdx.x; i < nt * vec_per_row; i += blockDim.x) {
      const int t = i / vec_per_row, v = i - t * vec_per_row;
      const __nv_bfloat16 *src;
      if (DOWN) {
        src = a.h + (size_t)(off + c0 + t) * a.I;
      } else {
        const int pair = a.plan.perm[off + c0 + t];
        src = a.x + (size_t)(pair / a.k) * a.H;
      }
      reinterpret_cast<uint4 *>(xs + (size_t)t * K)[v] = __ldg(reinterpret_cast<const uint4 *>(src) + v);
    }
    __syncthreads();
    if constexpr (!DOWN) {
      __nv_bfloat16 *hp = a.h + (size_t)(off + c0) * a.I;
      if (nt == 1) gateup_rows<FMT, 1>(blob, L, a.H, a.I, row0, xs, nt, hp, gs0, gs1);
      else if (nt == 2) gateup_rows<FMT, 2>(blob, L, a.H, a.I, row0, xs, nt, hp, gs0, gs1);
      else if (nt <= 4) gateup_rows<FMT, 4>(blob, L, a.H, a.I, row0, xs, nt, hp, gs0, gs1);
      else gateup_rows<FMT, 8>(blob, L, a.H, a.I, row0, xs, nt, hp, gs0, gs1);
    } else {
      float *yp = a.y + (size_t)(off + c0) * a.H;
      if (nt == 1) down_rows<FMT, 1>(blob, L, a.H, a.I, row0, xs, nt, yp, gs0);
      else if (nt == 2) down_rows<FMT, 2>(blob, L, a.H, a.I, row0, xs, nt, yp, gs0);
      else if (nt <= 4) down_rows<FMT, 4>(blob, L, a.H, a.I, row0, xs, nt, yp, gs0);
      else down_rows<FMT, 8>(blob, L, a.H, a.I, row0, xs, nt, yp, gs0);
    }
    __syncthreads();
  }
}

// Tokens with fewer than 8 rows staged leave rows nt..NT-1 of xs stale; the
// dot products of those rows are computed and dropped (lane == t < nt).

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

template <bool DOWN>
cudaError_t launch_ffn(const FfnArgs &a, cudaStream_t s) {
  const int rows = DOWN ? a.H : a.I;
  const int K = DOWN ? a.I : a.H;
  dim3 grid((rows + kRowsPerCta - 1) / kRowsPerCta, a.umax);
  const size_t smem = (size_t)kTokChunk * K * sizeof(__nv_bfloat16);
  switch (a.fmt) {
    case FMT_BF16: ffn_gemv_kernel<FMT_BF16, DOWN><<<grid, kFfnThreads, smem, s>>>(a); break;
    case FMT_NVFP4: ffn_gemv_kernel<FMT_NVFP4, DOWN><<<grid, kFfnThreads, smem, s>>>(a); break;
    default: ffn_gemv_kernel<FMT_MXFP4, DOWN><<<grid, kFfnThreads, smem, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

void ffn_init_attributes() {
  const int max_smem = kTokChunk * 8192 * 2;
  cudaFuncSetAttribute(ffn_gemv_kernel<FMT_BF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(ffn_gemv_kernel<FMT_NVFP4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(ffn_gemv_kernel<FMT_MXFP4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(ffn_gemv_kernel<FMT_BF16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(ffn_gemv_kernel<FMT_NVFP4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(ffn_gemv_kernel<FMT_MXFP4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

cudaError_t launch_gateup(const FfnArgs &a, cudaStream_t s) { return launch_ffn<false>(a, s); }
cudaError_t launch_down(const FfnArgs &a, cudaStream_t s) { return launch_ffn<true>(a, s); }

cudaError_t launch_combine(const float *y, const float *gates, const int32_t *inv, int T, int k, int H,
                           __nv_bfloat16 *out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dim3 grid((H / 4 + 255) / 256, T);
  combine_kernel<<<grid, 256, 0, s>>>(y, gates, inv, k, H, out);
  return cudaGetLastError();
}

}  // namespace ftmoe
