// gemv_dev.cuh -- device code of the decode expert FFN (dequant-fused GEMV)
// and of the combine fused into it, shared by the GEMV kernels and the fused
// decode layer kernel.  See ffn_gemv.cu for the design.
#pragma once
#include "ft_internal.cuh"
#include "wait_dev.cuh"

namespace ftmoe {
namespace {


constexpr int kWarps = 4;                       // per CTA
constexpr int kTokChunk = 4;                    // tokens per pass over the weights
constexpr int kMinFeatPerCta = kWarps;          // LPR = 32: one feature per warp
constexpr int kFusedCombineMaxT = 16;

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

// Raw bytes of one 32-element chunk of a weight row: FP4 = 16 code bytes +
// scale bits; FP8 = 32 code bytes (its scale is per row); BF16 = 64 bytes.
template <int FMT>
constexpr int chunk_vecs() { return FMT == FMT_BF16 ? 4 : FMT == FMT_FP8 ? 2 : 1; }
template <int FMT>
struct Chunk {
  uint4 q[chunk_vecs<FMT>()];
  uint32_t sf;
};

// Weight loads.  COH = false: the read-only path (ld.global.nc), for bytes
// that no one writes while the kernel runs (cached experts, pinned host
// memory).  COH = true: loads cached in L2 only (ld.global.cg), for a miss
// whose slot is filled while the kernel runs (by copying CTAs of the same
// grid, by the copy engine, or by CTAs that pull it from host memory); the
// flag wait before them orders them after those writes.
template <bool COH, typename T>
__device__ __forceinline__ T ld_w(const T *p) {
  if constexpr (COH) return __ldcg(p);
  else return __ldg(p);
}

template <int FMT, bool COH>
__device__ __forceinline__ void load_chunk(const uint8_t *__restrict__ codes_row,
                                           const uint8_t *__restrict__ sf_row, int c, Chunk<FMT> &ch) {
  if constexpr (FMT == FMT_BF16 || FMT == FMT_FP8) {
    constexpr int V = chunk_vecs<FMT>();
    const uint4 *p = reinterpret_cast<const uint4 *>(codes_row) + V * c;
#pragma unroll
    for (int i = 0; i < V; ++i) ch.q[i] = ld_w<COH>(p + i);
    ch.sf = 0;
  } else {
    ch.q[0] = ld_w<COH>(reinterpret_cast<const uint4 *>(codes_row) + c);
    if constexpr (FMT == FMT_NVFP4) ch.sf = ld_w<COH>(reinterpret_cast<const uint16_t *>(sf_row) + c);
    else ch.sf = ld_w<COH>(sf_row + c);
  }
}

// Decodes 8 weights (elements 8i .. 8i+7) of a chunk into w[8]: BF16 values,
// or the bare e2m1 values of FP4 codes (block scales are applied per 8-element
// partial sum, see chunk_fma).
template <int FMT>
__device__ __forceinline__ void decode8(const Chunk<FMT> &ch, int i, float *w) {
  if constexpr (FMT == FMT_BF16) {
    bf16x8_to_float(ch.q[i], w);
  } else if constexpr (FMT == FMT_FP8) {
    // eight E4M3 codes: bytes 8i .. 8i+7 of the chunk (exact in f16)
    const uint4 &v = ch.q[i >> 1];
    const uint32_t lo = (i & 1) ? v.z : v.x, hi = (i & 1) ? v.w : v.y;
    const uint32_t pairs[4] = {lo & 0xFFFFu, lo >> 16, hi & 0xFFFFu, hi >> 16};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 f = __half22float2(e4m3x2_to_half2(pairs[b]));
      w[2 * b] = f.x;
      w[2 * b + 1] = f.y;
    }
  } else {
    const uint32_t word = i == 0 ? ch.q[0].x : i == 1 ? ch.q[0].y : i == 2 ? ch.q[0].z : ch.q[0].w;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 v = __half22float2(e2m1x2_to_half2(word >> (8 * b)));
      w[2 * b] = v.x;
      w[2 * b + 1] = v.y;
    }
  }
}

// Position of 16-byte group q of a staged activation row: XOR-swizzled inside
// each 128-byte block, so that the lanes of a row group (which read groups
// 4c + i for consecutive chunks c) hit distinct banks.
__device__ __forceinline__ int xs_pos(int q) { return q ^ ((q >> 3) & 7); }

// c + a.lo * b.lo, then + a.hi * b.hi, for two pairs of 16-bit operands (bf16
// when BF, else f16) held in 32-bit words: each product is exact in fp32 and
// rounded once with its sum, as fmaf on the widened operands would be.
template <bool BF>
__device__ __forceinline__ float fma2x16(uint32_t a, uint32_t b, float c) {
  float d;
  if constexpr (BF)
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;\n\tfma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
  else
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %3;\n\tfma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
  return d;
}

// Activation row of a one-token pass (NT = 1), staged for multiplies on the
// 16-bit operands themselves (no conversion per product): BF16 weights take
// the bf16 row as it is; the other formats, whose codes convert to f16, take
// it as f16 scaled by a power of two s that puts the row's largest magnitude
// in [2^14, 2^15).  Every element down to 2^-31 of that largest one converts
// exactly, and the factor s passes exactly through every product and sum,
// so the dot products times 1/s (stored as a float after the row's K
// values) equal those of the unscaled fp32 arithmetic.  A row whose largest
// magnitude is zero or not finite is not scaled.  Every thread of the CTA
// calls this; the caller's barrier publishes the row.
template <int FMT, bool COH>
__device__ __forceinline__ void stage_row1(void *xs, const __nv_bfloat16 *src, int K) {
  const int nv = K / 8;
  uint4 *dst = reinterpret_cast<uint4 *>(xs);
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
  if constexpr (FMT == FMT_BF16) {
    for (int v = threadIdx.x; v < nv; v += blockDim.x) dst[xs_pos(v)] = ld_w<COH>(s4 + v);
  } else {
    __shared__ uint32_t s_wmax[32];
    uint32_t m = 0;   // largest |x| as fp32 bits
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      const uint4 q = ld_w<COH>(s4 + v);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) m = max(m, max((w[j] & 0x7FFFu) << 16, w[j] & 0x7FFF0000u));
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) s_wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = max(m, s_wmax[i]);
    int k = 0;
    if (m != 0 && m < 0x7F800000u) k = min(126, max(-126, 14 - ((int)(m >> 23) - 127)));
    const float s = __uint_as_float((uint32_t)(127 + k) << 23);
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      float f[8];
      bf16x8_to_float(ld_w<COH>(s4 + v), f);
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h = __floats2half2_rn(f[2 * j] * s, f[2 * j + 1] * s);
        o[j] = *reinterpret_cast<const uint32_t *>(&h);
      }
      dst[xs_pos(v)] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (threadIdx.x == 0)
      *reinterpret_cast<float *>(static_cast<char *>(xs) + (size_t)K * 2) = __uint_as_float((uint32_t)(127 - k) << 23);
  }
}

// Eight weights (elements 8i .. 8i+7 of a chunk) as four f16x2 words (FP4:
// bare e2m1 values; FP8: E4M3 values; both exact in f16).
template <int FMT>
__device__ __forceinline__ void decode8h(const Chunk<FMT> &ch, int i, uint32_t *w) {
  if constexpr (FMT == FMT_FP8) {
    const uint4 &v = ch.q[i >> 1];
    const uint32_t lo = (i & 1) ? v.z : v.x, hi = (i & 1) ? v.w : v.y;
    const uint32_t pairs[4] = {lo & 0xFFFFu, lo >> 16, hi & 0xFFFFu, hi >> 16};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const __half2 h = e4m3x2_to_half2(pairs[b]);
      w[b] = *reinterpret_cast<const uint32_t *>(&h);
    }
  } else {
    const uint32_t word = i == 0 ? ch.q[0].x : i == 1 ? ch.q[0].y : i == 2 ? ch.q[0].z : ch.q[0].w;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const __half2 h = e2m1x2_to_half2(word >> (8 * b));
      w[b] = *reinterpret_cast<const uint32_t *>(&h);
    }
  }
}

// acc[t] += chunk . xs[t][32c .. 32c+31].  FP4: each 8-element partial sum of
// e2m1 value x activation (every product exact in fp32) is multiplied by its
// block scale once (NVFP4: elements 0..15 and 16..31 have one E4M3 scale
// each; MXFP4: one E8M0 scale for all 32); the NVFP4 global scale is applied
// to the finished dot product.  One-token passes (NT = 1) multiply the 16-bit
// weights and staged activations directly (see stage_row1), in the same order.
template <int FMT, int NT>
__device__ __forceinline__ void chunk_fma(const Chunk<FMT> &ch, const __nv_bfloat16 *xs, int K, int c, int nt,
                                          float *acc) {
  float s0 = 1.0f, s1 = 1.0f;
  if constexpr (FMT == FMT_NVFP4) {
    const float2 s = __half22float2(e4m3x2_to_half2(ch.sf));
    s0 = s.x;
    s1 = s.y;
  } else if constexpr (FMT == FMT_MXFP4) {
    s0 = s1 = e8m0_to_float(ch.sf);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float s = i < 2 ? s0 : s1;
    if constexpr (NT == 1) {
      const uint4 xv = reinterpret_cast<const uint4 *>(xs)[xs_pos(4 * c + i)];
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t ww[4];
      if constexpr (FMT == FMT_BF16) {
        ww[0] = ch.q[i].x; ww[1] = ch.q[i].y; ww[2] = ch.q[i].z; ww[3] = ch.q[i].w;
      } else {
        decode8h<FMT>(ch, i, ww);
      }
      float p = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) p = fma2x16<FMT == FMT_BF16>(ww[j], xw[j], p);
      acc[0] = (FMT == FMT_BF16 || FMT == FMT_FP8) ? acc[0] + p : fmaf(s, p, acc[0]);
      continue;
    }
    float w[8];
    decode8<FMT>(ch, i, w);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t > 0 && t >= nt) break;   // uniform across the CTA: the expert's token rows in this pass
      const uint4 xv = reinterpret_cast<const uint4 *>(xs + (size_t)t * K)[xs_pos(4 * c + i)];
      float xf[8];
      bf16x8_to_float(xv, xf);
      float p = 0.0f;
#pragma unroll
      for (int q = 0; q < 8; ++q) p = fmaf(w[q], xf[q], p);
      acc[t] = (FMT == FMT_BF16 || FMT == FMT_FP8) ? acc[t] + p : fmaf(s, p, acc[t]);
    }
  }
}

// Sum over the LPR lanes of this lane's row group (xor stays inside the group).
template <int LPR>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct RowPtrs {
  const uint8_t *codes, *sf;
};

// Row r of W_gu (r < 2I) or of W_d, inside one blob.
template <int FMT>
__device__ __forceinline__ RowPtrs row_ptrs(const uint8_t *blob, const BlobLayout &L, bool down, int r, int K) {
  RowPtrs p;
  if constexpr (FMT == FMT_BF16) {
    p.codes = blob + (down ? L.d_codes : L.gu_codes) + (size_t)r * K * 2;
    p.sf = nullptr;
  } else if constexpr (FMT == FMT_NVFP4) {
    p.codes = blob + (down ? L.d_codes : L.gu_codes) + (size_t)r * (K / 2);
    p.sf = blob + (down ? L.d_sf : L.gu_sf) + (size_t)r * (K / 16);
  } else if constexpr (FMT == FMT_FP8) {
    p.codes = blob + (down ? L.d_codes : L.gu_codes) + (size_t)r * K;
    p.sf = blob + (down ? L.d_sf : L.gu_sf) + (size_t)r * 4;   // the row's fp32 scale
  } else {
    p.codes = blob + (down ? L.d_codes : L.gu_codes) + (size_t)r * (K / 2);
    p.sf = blob + (down ? L.d_sf : L.gu_sf) + (size_t)r * (K / 32);
  }
  return p;
}

// Dot products of NROWS weight rows (gate/up: 2, down: 1) with NT staged
// activation rows, over this lane's chunks l, l+LPR, l+2 LPR, ... of K.  Loads
// of a batch of chunks are all issued before any of them is used.
// Writes a chunk's raw bytes (codes and its block-scale bytes) to row `dst`.
template <int FMT>
__device__ __forceinline__ void store_chunk(const RowPtrs &dst, int c, const Chunk<FMT> &ch) {
  if constexpr (FMT == FMT_BF16 || FMT == FMT_FP8) {
    // (FP8 row scales are not part of a chunk: FT_MISS_PULL does not take FP8)
    constexpr int V = chunk_vecs<FMT>();
    uint4 *p = reinterpret_cast<uint4 *>(const_cast<uint8_t *>(dst.codes)) + V * c;
#pragma unroll
    for (int i = 0; i < V; ++i) p[i] = ch.q[i];
  } else {
    reinterpret_cast<uint4 *>(const_cast<uint8_t *>(dst.codes))[c] = ch.q[0];
    if constexpr (FMT == FMT_NVFP4) reinterpret_cast<uint16_t *>(const_cast<uint8_t *>(dst.sf))[c] = (uint16_t)ch.sf;
    else const_cast<uint8_t *>(dst.sf)[c] = (uint8_t)ch.sf;
  }
}

// With `dst` set (a miss read from host memory), every chunk read is also
// written to the same place in the expert's GPU slot.
template <int FMT, int NT, int NROWS, int LPR, bool COH>
__device__ __forceinline__ void rows_dot(const RowPtrs *rp, const RowPtrs *dst, int K, const __nv_bfloat16 *xs,
                                         int l8, int nt, float (&acc)[NROWS][NT]) {
  // a lane's chunks of a row in flight at once: all of them for rows of up to
  // 4 chunks per lane on one token; 2 when several token rows already hold
  // registers (more would cost occupancy)
  constexpr int kBatch = NT == 1 ? 4 : 2;
  const int cpl = K / (32 * LPR);  // chunks per lane
#pragma unroll 1
  for (int i0 = 0; i0 < cpl; i0 += kBatch) {
    Chunk<FMT> ch[NROWS][kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
      if (i0 + b < cpl)
#pragma unroll
        for (int r = 0; r < NROWS; ++r) load_chunk<FMT, COH>(rp[r].codes, rp[r].sf, l8 + LPR * (i0 + b), ch[r][b]);
    if (dst) {
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        if (i0 + b < cpl)
#pragma unroll
          for (int r = 0; r < NROWS; ++r) store_chunk<FMT>(dst[r], l8 + LPR * (i0 + b), ch[r][b]);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
      if (i0 + b < cpl)
#pragma unroll
        for (int r = 0; r < NROWS; ++r) chunk_fma<FMT, NT>(ch[r][b], xs, K, l8 + LPR * (i0 + b), nt, acc[r]);
  }
}

template <int FMT, bool DOWN, int NT, int LPR, bool COH>
__device__ __forceinline__ void ffn_rows(const uint8_t *blob, uint8_t *slot_dst, const BlobLayout &L, const FfnArgs &a,
                                         int feat, const __nv_bfloat16 *xs, int nt, int p0, float gs0, float gs1,
                                         int l8) {
  if constexpr (!DOWN) {
    if (feat >= a.I) return;
    const RowPtrs rp[2] = {row_ptrs<FMT>(blob, L, false, feat, a.H), row_ptrs<FMT>(blob, L, false, a.I + feat, a.H)};
    RowPtrs dp[2];
    if (slot_dst) {
      dp[0] = row_ptrs<FMT>(slot_dst, L, false, feat, a.H);
      dp[1] = row_ptrs<FMT>(slot_dst, L, false, a.I + feat, a.H);
    }
    float acc[2][NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[0][t] = acc[1][t] = 0.0f;
    if constexpr (FMT == FMT_FP8) {
      gs0 *= ld_w<COH>(reinterpret_cast<const float *>(rp[0].sf));
      gs1 *= ld_w<COH>(reinterpret_cast<const float *>(rp[1].sf));
    }
    rows_dot<FMT, NT, 2, LPR, COH>(rp, slot_dst ? dp : nullptr, a.H, xs, l8, nt, acc);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float g = group_sum<LPR>(acc[0][t]) * gs0;
      const float u = group_sum<LPR>(acc[1][t]) * gs1;
      if (l8 == t && t < nt) a.h[(size_t)(p0 + t) * a.I + feat] = __float2bfloat16_rn(g / (1.0f + expf(-g)) * u);
    }
  } else {
    if (feat >= a.H) return;
    const RowPtrs rp[1] = {row_ptrs<FMT>(blob, L, true, feat, a.I)};
    RowPtrs dp[1];
    if (slot_dst) dp[0] = row_ptrs<FMT>(slot_dst, L, true, feat, a.I);
    float acc[1][NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[0][t] = 0.0f;
    if constexpr (FMT == FMT_FP8) gs0 *= ld_w<COH>(reinterpret_cast<const float *>(rp[0].sf));
    rows_dot<FMT, NT, 1, LPR, COH>(rp, slot_dst ? dp : nullptr, a.I, xs, l8, nt, acc);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float v = group_sum<LPR>(acc[0][t]) * gs0;
      if (l8 == t && t < nt) a.y[(size_t)(p0 + t) * a.H + feat] = v;
    }
  }
}

// Work of one CTA (KW warps) on one (distinct expert u, feature block bx):
// KW * 32 / LPR * fpw output features, all of the expert's tokens, NT (>= the
// tokens any expert of the call has, up to kTokChunk) token rows per pass.
// xs: shared memory for NT activation rows of K.
// x_staged (gate/up of a one-token call): xs already holds the token's row.
// COH: every weight and activation load goes through L2 (ld.global.cg), for
// grids during which slots of misses (or h) are written; otherwise weights
// take the read-only path.
template <int FMT, bool DOWN, int NT, int LPR, int KW, bool COH>
__device__ __forceinline__ void gemv_block(const FfnArgs &a, int u, int bx, int fpw, __nv_bfloat16 *xs,
                                           bool x_staged = false) {
  // fpw passes per warp over feature groups: long rows (large K) give each CTA
  // more features, so that the staged activations serve more weight bytes
  const int kFeatPerCta = KW * (32 / LPR) * fpw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, l8 = lane & (LPR - 1);
  // the count and this item's packed plan entry, in one round trip (entries
  // past the count are stale and ignored)
  // (COH: the plan was written by a CTA of the same grid, so it is read through L2)
  const int nU = COH ? __ldcg(a.plan.n) : a.plan.n[0];
  const int4 ui = COH ? __ldcg(a.plan.u_info + u) : a.plan.u_info[u];
  const int hit = ui.w & 1;
  bool work = u < nU;
  if (work && ((a.only == 1 && !hit) || (a.only == 2 && hit))) work = false;
  if (work && !DOWN && !hit && a.copy_rows > 0) {
    // the copying CTAs of this grid raise the flag once every miss's gate/up bytes have landed
    __shared__ int s_ok;
    if (!cta_wait_flag(a.copy_sync, a.seq, a.err, 70, &s_ok)) return;
  }
  if (work) {
    const int e = ui.x;
    const int off = ui.z;
    const int n = ui.w >> 1;
    uint8_t *slot = const_cast<uint8_t *>(a.slot_bank) + (size_t)ui.y * a.slot_stride;
    const uint8_t *blob = slot;
    uint8_t *pull_dst = nullptr;
    if (a.pull && !hit) {
      // a miss read straight from pinned host memory over PCIe; the bytes read
      // are also written into its slot, so later calls hit
      blob = reinterpret_cast<const uint8_t *>(a.pool_dev[(size_t)a.layer * a.E + e]);
      pull_dst = slot;
    }
    const BlobLayout L = blob_layout(FMT, a.H, a.I);
    const int K = DOWN ? a.I : a.H;
    float gs0 = 1.0f, gs1 = 1.0f;
    if constexpr (FMT == FMT_NVFP4) {
      const float *gs = reinterpret_cast<const float *>(blob + L.gscale);
      if (!DOWN && !hit && a.ms.n > 0) {
        // the slot still waits for its down part, which holds the global scales
        for (int i = 0; i < a.ms.n; ++i)
          if (a.ms.expert[i] == e) {
            gs0 = a.ms.gate[i];
            gs1 = a.ms.up[i];
          }
      } else {
        gs0 = ld_w<COH>(gs + (DOWN ? 2 : 0));
        gs1 = ld_w<COH>(gs + 1);
      }
      if (DOWN && pull_dst && bx == 0 && threadIdx.x == 0)
        *reinterpret_cast<uint4 *>(pull_dst + L.gscale) = *reinterpret_cast<const uint4 *>(blob + L.gscale);
    }
    const int feat0 = bx * kFeatPerCta + warp * (32 / LPR) + lane / LPR;
    {
      // ask L2 for this lane's weight chunks now, so that their DRAM latency
      // overlaps the activation staging below
      const int cpl = K / (32 * LPR);
      const int cbytes = 16 * chunk_vecs<FMT>();
      for (int fp = 0; fp < fpw; ++fp) {
        const int feat = feat0 + fp * KW * (32 / LPR);
        if (feat >= (DOWN ? a.H : a.I)) break;
#pragma unroll
        for (int r = 0; r < (DOWN ? 1 : 2); ++r) {
          const RowPtrs rp = row_ptrs<FMT>(blob, L, DOWN, DOWN ? feat : (r == 0 ? feat : a.I + feat), K);
          for (int i = 0; i < cpl; ++i) {
            const uint8_t *p = rp.codes + (size_t)(l8 + LPR * i) * cbytes;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
          }
        }
      }
    }
    for (int c0 = 0; c0 < n; c0 += kTokChunk) {
      const int nt = min(kTokChunk, n - c0);
      // stage the chunk's activations in shared memory: one-token passes
      // through stage_row1, else bf16 rows of K
      if (NT == 1 && !x_staged) {
        const __nv_bfloat16 *src;
        if (DOWN) {
          src = a.h + (size_t)(off + c0) * a.I;
        } else {
          const int pair = COH ? __ldcg(a.plan.perm + off + c0) : a.plan.perm[off + c0];
          src = a.x + (size_t)(pair / a.k) * a.H;
        }
        stage_row1<FMT, COH>(xs, src, K);
      }
      const int vec_per_row = K / 8;
      for (int i = threadIdx.x; i < (NT == 1 || x_staged ? 0 : nt * vec_per_row); i += blockDim.x) {
        const int t = i / vec_per_row, v = i - t * vec_per_row;
        const __nv_bfloat16 *src;
        if (DOWN) {
          src = a.h + (size_t)(off + c0 + t) * a.I;
        } else {
          const int pair = COH ? __ldcg(a.plan.perm + off + c0 + t) : a.plan.perm[off + c0 + t];
          src = a.x + (size_t)(pair / a.k) * a.H;
        }
        reinterpret_cast<uint4 *>(xs + (size_t)t * K)[xs_pos(v)] = ld_w<COH>(reinterpret_cast<const uint4 *>(src) + v);
      }
      __syncthreads();
      // one-token passes on f16 activations: their scale comes off with the weights' own
      float g0 = gs0, g1 = gs1;
      if constexpr (NT == 1 && FMT != FMT_BF16) {
        const float inv = *reinterpret_cast<const float *>(reinterpret_cast<const char *>(xs) + (size_t)K * 2);
        g0 *= inv;
        g1 *= inv;
      }
      // rows nt..NT-1 of xs may hold stale data: their products are skipped
      for (int fp = 0; fp < fpw; ++fp)
        ffn_rows<FMT, DOWN, NT, LPR, COH>(blob, c0 == 0 ? pull_dst : nullptr, L, a, feat0 + fp * KW * (32 / LPR), xs,
                                          nt, off + c0, g0, g1, l8);
      __syncthreads();
    }
  }
}

// L2 prefetch of the weight rows of work item (u, bx) (a hit, or every
// expert when `any`): lets a CTA request all of its items' rows up front.
template <int FMT, bool DOWN, int LPR, int KW>
__device__ __forceinline__ void gemv_prefetch(const FfnArgs &a, int u, int bx, int fpw, bool any) {
  if (u >= a.plan.n[0]) return;
  const int4 ui = a.plan.u_info[u];
  if (!any && !(ui.w & 1)) return;
  const uint8_t *blob = a.slot_bank + (size_t)ui.y * a.slot_stride;
  const BlobLayout L = blob_layout(FMT, a.H, a.I);
  const int K = DOWN ? a.I : a.H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, l8 = lane & (LPR - 1);
  const int kFeatPerCta = KW * (32 / LPR) * fpw;
  const int feat0 = bx * kFeatPerCta + warp * (32 / LPR) + lane / LPR;
  const int cpl = K / (32 * LPR);
  const int cbytes = 16 * chunk_vecs<FMT>();
  for (int fp = 0; fp < fpw; ++fp) {
    const int feat = feat0 + fp * KW * (32 / LPR);
    if (feat >= (DOWN ? a.H : a.I)) break;
#pragma unroll
    for (int r = 0; r < (DOWN ? 1 : 2); ++r) {
      const RowPtrs rp = row_ptrs<FMT>(blob, L, DOWN, DOWN ? feat : (r == 0 ? feat : a.I + feat), K);
      for (int i = 0; i < cpl; ++i) {
        const uint8_t *p = rp.codes + (size_t)(l8 + LPR * i) * cbytes;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
      }
    }
  }
}

// Combine fused into the down projection: after its down work on feature
// block bx, a CTA counts itself done; the CTA that brings the count to
// `expected` writes out[t][f] = sum_j gates[t][j] * y[inv[t*k+j]][f] for the
// block's features (rank order j ascending) and resets the counter.
__device__ __forceinline__ void combine_block(const FfnArgs &a, const CombineArgs &cb, int bx, int feat_per_cta,
                                              int expected, int *s_flag) {
  // gates and positions of the call's (token, rank) pairs, read by every CTA
  // before the count so that the last one has them at hand
  __shared__ float s_g[kFusedCombineMaxT * kMaxTopK];
  __shared__ int s_inv[kFusedCombineMaxT * kMaxTopK];
  for (int i = threadIdx.x; i < cb.T * a.k; i += blockDim.x) {
    s_g[i] = __ldcg(cb.gates + i);
    s_inv[i] = __ldcg(cb.inv + i);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(cb.counters + bx, 1);
    *s_flag = prev == expected - 1;
  }
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();
  const int f0 = bx * feat_per_cta;
  for (int i = threadIdx.x; i < cb.T * feat_per_cta; i += blockDim.x) {
    const int t = i / feat_per_cta, f = f0 + (i - t * feat_per_cta);
    if (f >= a.H) continue;
    float acc = 0.0f;
    for (int j = 0; j < a.k; ++j)
      acc = fmaf(s_g[t * a.k + j], __ldcg(a.y + (size_t)s_inv[t * a.k + j] * a.H + f), acc);
    cb.out[(size_t)t * a.H + f] = __float2bfloat16_rn(acc);
  }
  if (threadIdx.x == 0) cb.counters[bx] = 0;
}

}  // namespace
}  // namespace ftmoe
