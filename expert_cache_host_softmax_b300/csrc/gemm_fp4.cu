// gemm_fp4.cu -- the FP4 x FP4 variant of the prefill expert FFN: NVFP4 weights
// times NVFP4-quantised activations on the block-scaled tensor cores
// (tcgen05.mma kind::mxf4nvf4, E2M1 operands, one E4M3 scale per 16 elements
// of each operand row, fp32 accumulators in TMEM).
//
// "FreeToken: Run Frontier MoE Models on Your Own GPU, and the RAM It Takes",
// section "The Real Requirement Is System RAM": NVFP4 is 4-bit values plus an
// 8-bit scale per 16 weights.  The pages say nothing of activation precision;
// this variant quantises x and h to the same layout so that both GEMM operands
// are FP4 (the weight-only path in grouped_gemm.cu keeps bf16 activations).
//
// Activation quantiser (all decisions in IEEE binary32):
//   x rows: g = amax(row) / (6 * 448) (1 for an all-zero row),
//           s_b = E4M3_rn((amax(block of 16) / 6) / g),
//           r_b = 1 / (value(s_b) * g)  (one rounding; 0 where the product is 0),
//           q = e2m1_rn(x * r_b)
//   h rows: the same with g = 1 (the E4M3 block scales alone).
// x is quantised once per token and scattered to its k (token, rank) pairs in
// an expert-padded row order: expert e's rows start at pad_start[e] =
// sum over e' < e of ceil(count(e') / 128) * 128, so every 128-row tile of an
// expert is one aligned block of rows and of scale-factor atoms.  Rows past an
// expert's count are never written; their products are never stored.
//
// Scale factors go to TMEM in the layout the block-scaled MMA reads: per 128
// rows and 4 blocks of 16 (one MMA's K of 64), a 512-byte atom in which byte
// 16*(r % 32) + 4*(r / 32) + b holds row r's block b, copied with
// tcgen05.cp.32x128b.warpx4 into 4 TMEM columns.  The quantisers write x's and
// h's scales in that atom order in global memory; the weights' scales (row
// order in the blob) are re-ordered into it by one warp per stage.
//
// One persistent CTA per SM walks 128 x 128 output tiles (gate/up: 64 gate
// rows + the 64 matching up rows, so the epilogue has both halves of 64 h
// columns; down: 128 rows of H), K in stages of 256 (128 bytes of codes a row):
//   warp 0   producer: TMA of the A box (128 padded rows x 128 bytes, 128-byte
//            swizzle), of the B box(es) from the slot bank, and a bulk copy of
//            the stage's A scale atoms (2 KB);
//   warp 1   MMA: tcgen05.cp of the stage's scale atoms, 4 MMAs of K = 64
//            (M = 128, N = 128) into one of two TMEM accumulators;
//   warp 2   B scales: the producer's TMA lands the tile rows' scale bytes in
//            row order (16 bytes a row per stage); this warp stores them as atoms;
//   warps 4-11 epilogue, one TMEM lane (tile row) per thread, two warps per
//            lane quarter (each half of the tile's columns): gate/up applies
//            the row's x scale and the NVFP4 global scales, SiLU * up, and
//            quantises h (block scales, codes in padded order); down applies
//            the global scale and adds gate * y into the token's fp32 output
//            row (the combine), storing y when asked.
// Every wait is bounded, as in grouped_gemm.cu.
#include <cuda.h>

#include <algorithm>

#include "ft_internal.cuh"
#include "tc_ptx.cuh"

namespace ftmoe {

namespace {

using namespace tc;

constexpr int QBM = 128;              // padded rows per tile (one TMEM lane each)
constexpr int QBN = 128;              // weight rows per tile (MMA N)
constexpr int QBK = 256;              // K elements per stage: 128 bytes of e2m1 codes a row
constexpr int QNS = 5;                // stages
constexpr int Q_A = QBM * QBK / 2;    // 16 KB
constexpr int Q_B = QBN * QBK / 2;    // 16 KB
constexpr int Q_SF = 128 * (QBK / 16);  // 2 KB: 4 atoms of 512 bytes
constexpr int Q_OFF_B = QNS * Q_A;
constexpr int Q_OFF_SFA = Q_OFF_B + QNS * Q_B;
constexpr int Q_OFF_SFB = Q_OFF_SFA + QNS * Q_SF;
constexpr int Q_OFF_SFR = Q_OFF_SFB + QNS * Q_SF;   // B scales as they sit in the blob (row order)
constexpr int Q_OFF_BAR = Q_OFF_SFR + QNS * Q_SF;
constexpr int Q_BARS = 3 * QNS + 5;   // FULL, EMPTY, SFRAW per stage; TFULL x2, TEMPTY x2, DRAIN
constexpr int Q_OFF_TAB = Q_OFF_BAR + Q_BARS * 8 + 16;
constexpr int Q_EPI_WARPS = 8;        // two per TMEM lane quarter, each half of a tile's columns
// down epilogue: one 32 x 16 fp32 transpose block per epilogue warp (rows padded to 20)
constexpr int Q_OFF_XP = (Q_OFF_TAB + 4 * 3 * (kMaxExperts + 1) + 64 + 15) / 16 * 16;
constexpr int Q_XP_STRIDE = 20;
constexpr int Q_SMEM = Q_OFF_XP + Q_EPI_WARPS * 32 * Q_XP_STRIDE * 4;
constexpr int Q_SMEM_ALLOC = Q_SMEM + 1024;
constexpr int Q_THREADS = (4 + Q_EPI_WARPS) * 32;
constexpr int Q_PROD = 0, Q_MMA = 1, Q_SFW = 2, Q_EPI0 = 4;
constexpr uint32_t Q_TMEM_COLS = 512;  // accumulators 0 and 128; scale buffers from 256
constexpr uint32_t Q_SFA_COL = 256, Q_SFB_COL = 288;   // + 16 * (stage parity)

// M = 128, N = 128, A and B E2M1 (format 1 of the mxf4 kinds), UE4M3 scales
// (bit 23 clear), K-major, dense K = 64.
constexpr uint32_t kIdescFp4 = (1u << 7) | (1u << 10) | ((uint32_t)(QBN >> 3) << 17) | ((uint32_t)(QBM >> 4) << 24);

static_assert(Q_SMEM_ALLOC <= 227 * 1024, "fp4 gemm smem");

// D[tmem] (+)= A . B^T with E2M1 operands, each row's blocks of 16 scaled by
// the UE4M3 factors at sfa / sfb (TMEM), fp32 accumulate.
__device__ __forceinline__ void mma_fp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// One 512-byte scale atom (32 lines of 16 bytes) from shared memory into 4
// TMEM columns of every lane quarter.
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;               // LBO (one 16-byte column: unused)
  d |= (uint64_t)(128 >> 4) << 32;      // SBO: 8-line groups 128 bytes apart
  d |= (uint64_t)1 << 46;               // descriptor version
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

// Bulk copy of `bytes` (multiple of 16) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// ---------------------------------------------------------------- quantiser

// Non-negative fp32 -> E4M3 code (nearest, ties to even, saturating at 448)
// and that code's value.
__device__ __forceinline__ uint32_t e4m3_rn(float s, float *val) {
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(s));
  const uint32_t code = pair & 0xFFu;
  *val = e4m3_to_float(code);
  return code;
}

// Two fp32 -> one byte of e2m1 codes (lo in bits 0-3), nearest, ties to even,
// saturating at 6 (the first source of the conversion fills the upper nibble).
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tmov.b16 %0, {b, b};\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

__device__ __forceinline__ void bf16x8_unpack(const uint4 &v, float *f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Quantises 16 values with the global scale g: returns the E4M3 scale code,
// writes 8 code bytes (element 2j in the low nibble of byte j) to q[0..1].
__device__ __forceinline__ uint32_t quant16(const float *v, float g, uint32_t *q) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  float sval;
  const uint32_t sc = e4m3_rn(__fdiv_rn(__fdiv_rn(amax, 6.0f), g), &sval);
  const float den = __fmul_rn(sval, g);
  const float r = den > 0.0f ? __frcp_rn(den) : 0.0f;
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i >> 2] |= e2m1x2_rn(__fmul_rn(v[2 * i], r), __fmul_rn(v[2 * i + 1], r)) << (8 * (i & 3));
  q[0] = w[0];
  q[1] = w[1];
  return sc;
}

// Byte offset of (padded row r, block b) in a scale-atom array of rows with
// K elements: atoms ordered by 128-row block, then by group of 4 blocks.
__device__ __forceinline__ size_t sf_atom_off(int r, int b, int K) {
  return ((size_t)(r >> 7) * (K >> 6) + (b >> 2)) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3) + (b & 3);
}

// First padded row of expert e: sum over e' < e of ceil(count(e') / 128) * 128.
__device__ __forceinline__ int warp_pad_start(const int32_t *offsets, int e) {
  const int lane = threadIdx.x & 31;
  int s = 0;
  for (int i = lane; i < e; i += 32) s += (offsets[i + 1] - offsets[i] + 127) & ~127;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// One CTA per token: quantise x[t] (row scale), then write its codes, block
// scales and row scale to the padded row of each of its k (token, rank) pairs.
__global__ void __launch_bounds__(128) quant_x_kernel(const __nv_bfloat16 *__restrict__ x,
                                                      const int32_t *__restrict__ topk_idx,
                                                      const int32_t *__restrict__ inv,
                                                      const int32_t *__restrict__ offsets, int k, int H,
                                                      uint8_t *__restrict__ xq, uint8_t *__restrict__ xsf,
                                                      float *__restrict__ xg) {
  __shared__ int s_prow[kMaxTopK];
  __shared__ float s_amax[4];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  // padded rows of the token's pairs
  for (int j = w; j < k; j += 4) {
    const int p = t * k + j, e = topk_idx[p];
    const int ps = warp_pad_start(offsets, e);
    if (lane == 0) s_prow[j] = ps + (inv[p] - offsets[e]);
  }
  const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
  const int nblk = H / 16;
  float amax = 0.0f;
  for (int b = tid; b < nblk; b += 128) {
    float v[16];
    bf16x8_unpack(__ldg(xr + 2 * b), v);
    bf16x8_unpack(__ldg(xr + 2 * b + 1), v + 8);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_amax[w] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(s_amax[0], s_amax[1]), fmaxf(s_amax[2], s_amax[3]));
  const float g = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
  for (int b = tid; b < nblk; b += 128) {
    float v[16];
    bf16x8_unpack(__ldg(xr + 2 * b), v);
    bf16x8_unpack(__ldg(xr + 2 * b + 1), v + 8);
    uint32_t q[2];
    const uint32_t sc = quant16(v, g, q);
    for (int j = 0; j < k; ++j) {
      const int r = s_prow[j];
      *reinterpret_cast<uint2 *>(xq + (size_t)r * (H / 2) + 8 * b) = make_uint2(q[0], q[1]);
      xsf[sf_atom_off(r, b, H)] = (uint8_t)sc;
    }
  }
  if (tid < k) xg[s_prow[tid]] = g;
}

// ---------------------------------------------------------------- GEMM

struct Fp4Args {
  const uint8_t *slot_bank;
  long long slot_stride;
  int H, I, k;
  PlanBufs plan;
  int only;                 // 0 all, 1 hits, 2 misses
  long long gscale_off;     // byte offset of the NVFP4 global scales in a blob
  const uint8_t *a_sf;      // A scale atoms (x or h)
  const float *xg;          // gate/up: row scale of each padded row
  uint8_t *hq;              // gate/up: h codes [rows][I/2]
  uint8_t *hsf;             // gate/up: h scale atoms
  float *y;                 // down: [T*k][H] (permuted order), when keep_y
  float *out_acc;           // down: out_acc[token] += gate * y row
  int keep_y;
  int *err;
};

struct QTile {
  int u, n, mt;
  int row0, rows;   // first permuted row, valid rows
  int prow0;        // first padded row
  int slot;
};

__device__ __forceinline__ QTile q_decode(int t, const int *s_start, const int *s_mt, const int *s_pad, int nU,
                                          int NTN, const Fp4Args &a) {
  int lo = 0, hi = nU;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_start[mid] * NTN <= t) lo = mid;
    else hi = mid;
  }
  QTile q;
  q.u = lo;
  const int mt = s_mt[lo];
  const int rem = t - s_start[lo] * NTN;
  q.n = rem / mt;
  q.mt = rem - q.n * mt;
  const int e = a.plan.u_expert[lo];
  const int off = a.plan.offsets[e], cnt = a.plan.offsets[e + 1] - off;
  q.row0 = off + q.mt * QBM;
  q.rows = min(QBM, cnt - q.mt * QBM);
  q.prow0 = (s_pad[lo] + q.mt) * QBM;
  q.slot = a.plan.u_slot[lo];
  return q;
}

template <bool DOWN>
__global__ void __launch_bounds__(Q_THREADS, 1)
    gemm_fp4_kernel(Fp4Args a, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmSB) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  unsigned char *sm = smem_raw + (base - raw_base);
  const uint32_t sA = base, sB = base + Q_OFF_B, sSFA = base + Q_OFF_SFA, sSFB = base + Q_OFF_SFB;
  const uint32_t sSFR = base + Q_OFF_SFR;
  const uint32_t bar0 = base + Q_OFF_BAR;
  auto FULL = [&](int s) { return bar0 + 8u * s; };
  auto EMPTY = [&](int s) { return bar0 + 8u * (QNS + s); };
  auto SFRAW = [&](int s) { return bar0 + 8u * (2 * QNS + s); };
  auto TFULL = [&](int b) { return bar0 + 8u * (3 * QNS + b); };
  auto TEMPTY = [&](int b) { return bar0 + 8u * (3 * QNS + 2 + b); };
  const uint32_t DRAIN = bar0 + 8u * (3 * QNS + 4);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + Q_OFF_BAR + Q_BARS * 8);
  volatile int *s_abort = reinterpret_cast<volatile int *>(sm + Q_OFF_BAR + Q_BARS * 8 + 4);
  int *s_start = reinterpret_cast<int *>(sm + Q_OFF_TAB);
  int *s_mt = s_start + (kMaxExperts + 1);
  int *s_pad = s_mt + (kMaxExperts + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = DOWN ? a.I : a.H;
  const int nk = K / QBK;
  const int NTN = DOWN ? a.H / QBN : a.I / (QBN / 2);

  if (tid == 0) {
    for (int s = 0; s < QNS; ++s) {
      mbar_init(FULL(s), 1 + 32);     // the producer's expect_tx + the B-scale warp's lanes
      mbar_init(EMPTY(s), 1);
      mbar_init(SFRAW(s), 1);         // the producer's expect_tx for the B scales in row order
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(TFULL(b), 1);
      mbar_init(TEMPTY(b), Q_EPI_WARPS * 32);
    }
    mbar_init(DRAIN, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == Q_MMA) tmem_alloc(smem_u32(s_tmem), Q_TMEM_COLS);
  const int nU = a.plan.n[0];
  if (warp == Q_EPI0) {
    // per distinct expert: M tiles of the selected experts (prefix in s_start)
    // and the padded row blocks of all experts (prefix in s_pad)
    int run = 0, prun = 0;
    for (int u0 = 0; u0 < nU; u0 += 32) {
      const int u = u0 + lane;
      int mt = 0, pb = 0;
      if (u < nU) {
        const int e = a.plan.u_expert[u];
        const int cnt = a.plan.offsets[e + 1] - a.plan.offsets[e];
        const int hit = a.plan.u_hit[u];
        const bool sel = a.only == 0 || (a.only == 1 && hit) || (a.only == 2 && !hit);
        pb = (cnt + QBM - 1) / QBM;
        mt = sel ? pb : 0;
        s_mt[u] = mt;
      }
      int x = mt, y = pb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int xs = __shfl_up_sync(0xffffffffu, x, o), ys = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) {
          x += xs;
          y += ys;
        }
      }
      if (u < nU) {
        s_start[u] = run + x - mt;
        s_pad[u] = prun + y - pb;
      }
      run += __shfl_sync(0xffffffffu, x, 31);
      prun += __shfl_sync(0xffffffffu, y, 31);
    }
    if (lane == 0) s_start[nU] = run;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int n_tiles = s_start[nU] * NTN;

  if (warp == Q_PROD) {
    // ================================================================ producer
    if (lane == 0) {
      int j = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const QTile ti = q_decode(tile, s_start, s_mt, s_pad, nU, NTN, a);
        const uint8_t *sfa = a.a_sf + (size_t)(ti.prow0 >> 7) * (K >> 6) * 512;
        for (int kb = 0; kb < nk; ++kb, ++j) {
          const int s = j % QNS;
          if (!mbar_wait(EMPTY(s), ((j / QNS) & 1) ^ 1, s_abort, a.err, 110)) { ok = false; break; }
          mbar_arrive_expect_tx(FULL(s), Q_A + Q_B + Q_SF);
          tma_load_2d(sA + s * Q_A, &tmA, FULL(s), kb * (QBK / 2), ti.prow0);
          if constexpr (DOWN) {
            tma_load_3d(sB + s * Q_B, &tmB, FULL(s), kb * (QBK / 2), ti.n * QBN, ti.slot);
          } else {
            tma_load_3d(sB + s * Q_B, &tmB, FULL(s), kb * (QBK / 2), ti.n * (QBN / 2), ti.slot);
            tma_load_3d(sB + s * Q_B + Q_B / 2, &tmB, FULL(s), kb * (QBK / 2), a.I + ti.n * (QBN / 2), ti.slot);
          }
          bulk_load(sSFA + s * Q_SF, sfa + (size_t)kb * Q_SF, Q_SF, FULL(s));
          // B scales in row order: 16 bytes (the stage's 16 blocks) of each tile row
          mbar_arrive_expect_tx(SFRAW(s), Q_SF);
          if constexpr (DOWN) {
            tma_load_3d(sSFR + s * Q_SF, &tmSB, SFRAW(s), kb * 16, ti.n * QBN, ti.slot);
          } else {
            tma_load_3d(sSFR + s * Q_SF, &tmSB, SFRAW(s), kb * 16, ti.n * (QBN / 2), ti.slot);
            tma_load_3d(sSFR + s * Q_SF + Q_SF / 2, &tmSB, SFRAW(s), kb * 16, a.I + ti.n * (QBN / 2), ti.slot);
          }
        }
      }
      // every copy this CTA issued must land before the CTA exits
      for (int jj = max(0, j - QNS); jj < j; ++jj) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(FULL(jj % QNS), (jj / QNS) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
        while (!mbar_try_wait(SFRAW(jj % QNS), (jj / QNS) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == Q_SFW) {
    // ================================================================ B scales
    // Lane l moves tile rows l, l+32, l+64, l+96 (16 bytes each: the stage's
    // 16 blocks) from row order into atom g's line l = {row l, row l+32,
    // row l+64, row l+96} x word g.
    int j = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      for (int kb = 0; kb < nk; ++kb, ++j) {
        const int s = j % QNS;
        if (!mbar_wait(SFRAW(s), (j / QNS) & 1, s_abort, a.err, 111)) { ok = false; break; }
        uint4 r[4];
        const uint32_t src = sSFR + s * Q_SF + 16 * lane;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(r[i].x), "=r"(r[i].y), "=r"(r[i].z), "=r"(r[i].w)
                       : "r"(src + 512 * i)
                       : "memory");
        const uint32_t dst = sSFB + s * Q_SF + 16 * lane;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(r[0].x), "r"(r[1].x), "r"(r[2].x),
                     "r"(r[3].x)
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 512), "r"(r[0].y), "r"(r[1].y),
                     "r"(r[2].y), "r"(r[3].y)
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 1024), "r"(r[0].z), "r"(r[1].z),
                     "r"(r[2].z), "r"(r[3].z)
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 1536), "r"(r[0].w), "r"(r[1].w),
                     "r"(r[2].w), "r"(r[3].w)
                     : "memory");
        fence_proxy_async();   // these stores are visible to the tensor core's copy
        mbar_arrive(FULL(s));
      }
    }
  } else if (warp == Q_MMA) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      int j = 0, tl = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tl) {
        const int b = tl & 1;
        if (!mbar_wait(TEMPTY(b), ((tl >> 1) & 1) ^ 1, s_abort, a.err, 120)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + b * QBN;
        for (int kb = 0; kb < nk; ++kb, ++j) {
          const int s = j % QNS;
          if (!mbar_wait(FULL(s), (j / QNS) & 1, s_abort, a.err, 121)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + Q_SFA_COL + 16 * (j & 1), sfb_t = tmem_base + Q_SFB_COL + 16 * (j & 1);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            tmem_cp_atom(sfa_t + 4 * g, sSFA + s * Q_SF + 512 * g);
            tmem_cp_atom(sfb_t + 4 * g, sSFB + s * Q_SF + 512 * g);
          }
          const uint32_t a0 = sA + s * Q_A, b0 = sB + s * Q_B;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            mma_fp4(d, sdesc_sw128(a0 + 32 * g), sdesc_sw128(b0 + 32 * g), kIdescFp4, sfa_t + 4 * g, sfb_t + 4 * g,
                    (kb | g) != 0);
          mma_commit(EMPTY(s));
        }
        if (ok) mma_commit(TFULL(b));
      }
      mma_commit(DRAIN);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(DRAIN, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else if (warp >= Q_EPI0) {
    // ================================================================ epilogue
    const int q = warp & 3;                   // TMEM lane quarter
    const int half = (warp - Q_EPI0) >> 2;    // which half of the tile's columns
    const int row = q * 32 + lane;
    int tl = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tl) {
      const int b = tl & 1;
      const QTile ti = q_decode(tile, s_start, s_mt, s_pad, nU, NTN, a);
      if (!mbar_wait(TFULL(b), (tl >> 1) & 1, s_abort, a.err, 130)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + b * QBN;
      const float *gs = reinterpret_cast<const float *>(a.slot_bank + (size_t)ti.slot * a.slot_stride + a.gscale_off);
      const bool valid = row < ti.rows;
      const int prow = ti.prow0 + row;
      if constexpr (!DOWN) {
        // this half: h columns 32*half .. +31 of the tile's 64 (gate column c, up column 64 + c)
        const float gx = valid ? a.xg[prow] : 0.0f;
        const float g0 = gs[0] * gx, g1 = gs[1] * gx;
        uint32_t codes[4];
        uint32_t scw = 0;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          const int c = 32 * half + 16 * cb;
          float gv[16], uv[16];
          tmem_ld16(tb + c, gv);
          tmem_ld16(tb + QBN / 2 + c, uv);
          float hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gg = gv[i] * g0, uu = uv[i] * g1;
            hv[i] = gg * __frcp_rn(1.0f + __expf(-gg)) * uu;
          }
          uint32_t qq[2];
          const uint32_t sc = quant16(hv, 1.0f, qq);
          codes[2 * cb] = qq[0];
          codes[2 * cb + 1] = qq[1];
          scw |= sc << (8 * cb);
        }
        if (valid) {
          // 32 h columns = 16 code bytes and 2 block scales
          *reinterpret_cast<uint4 *>(a.hq + (size_t)prow * (a.I / 2) + ti.n * 32 + 16 * half) =
              make_uint4(codes[0], codes[1], codes[2], codes[3]);
          *reinterpret_cast<uint16_t *>(a.hsf + sf_atom_off(prow, 4 * ti.n + 2 * half, a.I)) = (uint16_t)scw;
        }
      } else {
        const float g0 = gs[2];
        const int c0 = half * (QBN / 2);
        float *dst = a.y + (size_t)(ti.row0 + row) * a.H + ti.n * QBN + c0;
        float *acc = nullptr;
        float gw = 0.0f;
        if (a.out_acc != nullptr && valid) {
          const int pair = a.plan.perm[ti.row0 + row];
          acc = a.out_acc + (size_t)(pair / a.k) * a.H + ti.n * QBN + c0;
          gw = a.plan.gates[pair] * g0;
        }
        const bool store_y = a.out_acc == nullptr || a.keep_y;
        const uint64_t opol = l2_evict_last();   // the output rows stay in L2 for the other pairs' updates
        // the reductions go through a per-warp transpose (as in the bf16
        // grouped GEMM): instruction j covers rows 8 j .. 8 j + 7 of the
        // warp, four lanes a row, 64 contiguous bytes each
        float *xp = reinterpret_cast<float *>(sm + Q_OFF_XP) + (size_t)((warp - Q_EPI0) * 32) * Q_XP_STRIDE;
        float *racc[4];
        float rgw[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int src = 8 * jj + (lane >> 2);
          racc[jj] = reinterpret_cast<float *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(acc), src));
          rgw[jj] = __shfl_sync(0xffffffffu, gw, src);
        }
#pragma unroll 1
        for (int c = 0; c < QBN / 2; c += 16) {
          float v[16];
          tmem_ld16(tb + c0 + c, v);
          if (valid && store_y) {
            float4 *o = reinterpret_cast<float4 *>(dst + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              o[i] = make_float4(v[4 * i] * g0, v[4 * i + 1] * g0, v[4 * i + 2] * g0, v[4 * i + 3] * g0);
          }
          if (a.out_acc != nullptr) {
            float4 *w4 = reinterpret_cast<float4 *>(xp + lane * Q_XP_STRIDE);
#pragma unroll
            for (int i = 0; i < 4; ++i) w4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int r = 8 * jj + (lane >> 2), f4 = lane & 3;
              const float4 t = *reinterpret_cast<const float4 *>(xp + r * Q_XP_STRIDE + 4 * f4);
              if (racc[jj] != nullptr)
                red_add_v4(racc[jj] + c + 4 * f4,
                           make_float4(t.x * rgw[jj], t.y * rgw[jj], t.z * rgw[jj], t.w * rgw[jj]), opol);
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before();
      mbar_arrive(TEMPTY(b));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == Q_MMA) tmem_dealloc(tmem_base, Q_TMEM_COLS);
}

// ---------------------------------------------------------------- peak probe

// Tensor-pipe rate of the block-scaled FP4 MMA alone: every CTA issues
// `iters` x 4 MMAs (M = 128, N = n_tile, K = 64) on operands already in shared
// memory, committing each group of 4; operands and scales are fixed patterns.
template <int NT>
__global__ void __launch_bounds__(128, 1) fp4_peak_kernel(int iters, int *err) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  unsigned char *sm = smem_raw + (base - raw_base);
  const uint32_t sA = base, sB = base + Q_A, sSF = base + Q_A + NT * 128;
  const uint32_t bar = sSF + 2 * Q_SF;
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + (bar - base) + 16);
  const int tid = threadIdx.x, warp = tid >> 5;
  // operands: a fixed pattern of codes; scales: E4M3 1.0 (0x38)
  for (int i = tid; i < (Q_A + NT * 128) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t *>(sm)[i] = 0x21436587u * (uint32_t)(i + 1);
  for (int i = tid; i < 2 * Q_SF / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(sm + (sSF - base))[i] = 0x38383838u;
  fence_proxy_async();
  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(smem_u32(s_tmem), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  constexpr uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) | ((uint32_t)(QBM >> 4) << 24);
  if (tid == 0) {
#pragma unroll
    for (int g = 0; g < 4; ++g) tmem_cp_atom(tmem + 256 + 4 * g, sSF + 512 * g);
#pragma unroll
    for (int g = 0; g < NT / 32; ++g) tmem_cp_atom(tmem + 272 + 4 * g, sSF + Q_SF + 512 * (g & 3));
    for (int it = 0; it < iters; ++it)
#pragma unroll
      for (int g = 0; g < 4; ++g)
        mma_fp4(tmem, sdesc_sw128(sA + 32 * g), sdesc_sw128(sB + 32 * g), idesc, tmem + 256, tmem + 272,
                (it | g) != 0);
    mma_commit(bar);
    const unsigned long long t0 = globaltimer();
    bool done = false;
    while (!(done = mbar_try_wait(bar, 0)) && globaltimer() - t0 < kWaitLimitNs) {
    }
    if (!done) atomicCAS(err, 0, 140);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

// ---------------------------------------------------------------- host side

void fp4_init_attributes() {
  cudaFuncSetAttribute(gemm_fp4_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, Q_SMEM_ALLOC);
  cudaFuncSetAttribute(gemm_fp4_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Q_SMEM_ALLOC);
}

int64_t fp4_padded_rows(int64_t rows, int64_t umax) { return (rows + (int64_t)QBM * umax + QBM - 1) / QBM * QBM; }

cudaError_t launch_quant_x(const __nv_bfloat16 *x, const PlanBufs &plan, int T, int k, int H, uint8_t *xq,
                           uint8_t *xsf, float *xg, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  quant_x_kernel<<<T, 128, 0, s>>>(x, plan.topk_idx, plan.inv, plan.offsets, k, H, xq, xsf, xg);
  return cudaGetLastError();
}

cudaError_t launch_tc_ffn_fp4(const FfnArgs &f, bool down, const Fp4Bufs &q, const void *map_a, const void *map_b,
                              const void *map_sfb, int *err, int64_t max_rows, cudaStream_t s) {
  Fp4Args a{};
  a.slot_bank = f.slot_bank;
  a.slot_stride = f.slot_stride;
  a.H = f.H;
  a.I = f.I;
  a.k = f.k;
  a.plan = f.plan;
  a.only = f.only;
  const BlobLayout L = blob_layout(FMT_NVFP4, f.H, f.I);
  a.gscale_off = L.gscale;
  a.a_sf = down ? q.hsf : q.xsf;
  a.xg = q.xg;
  a.hq = q.hq;
  a.hsf = q.hsf;
  a.y = f.y;
  a.out_acc = down ? f.out_acc : nullptr;
  a.keep_y = f.keep_y;
  a.err = err;
  const int NTN = down ? f.H / QBN : f.I / (QBN / 2);
  const int64_t mtiles = (max_rows + QBM - 1) / QBM + f.umax;
  const int grid = (int)std::min<int64_t>(tc_num_sms(), std::max<int64_t>(1, mtiles * NTN));
  const CUtensorMap &mA = *reinterpret_cast<const CUtensorMap *>(map_a);
  const CUtensorMap &mB = *reinterpret_cast<const CUtensorMap *>(map_b);
  const CUtensorMap &mS = *reinterpret_cast<const CUtensorMap *>(map_sfb);
  if (down) gemm_fp4_kernel<true><<<grid, Q_THREADS, Q_SMEM_ALLOC, s>>>(a, mA, mB, mS);
  else gemm_fp4_kernel<false><<<grid, Q_THREADS, Q_SMEM_ALLOC, s>>>(a, mA, mB, mS);
  return cudaGetLastError();
}

// TMA maps of the FP4 x FP4 GEMMs: A = quantised activations [rows][K/2]
// (box 128 bytes x 128 rows), B = the slot bank's e2m1 codes of one matrix,
// 3-D (K/2, rows, slot) with a box of 128 bytes x (64 gate/up | 128 down) rows,
// all with the 128-byte swizzle; and the B matrices' block scales, 3-D
// (K/16, rows, slot) with a box of 16 bytes x (64 | 128) rows, no swizzle.
int make_fp4_maps(const uint8_t *slots, int64_t slot_stride, int S, int H, int I, const void *xq, const void *hq,
                  int64_t rows, void *map_xq, void *map_hq, void *map_gu, void *map_d, void *map_gu_sf,
                  void *map_d_sf) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return -1;
  const BlobLayout L = blob_layout(FMT_NVFP4, H, I);
  const cuuint32_t estr[3] = {1, 1, 1};
  for (int which = 0; which < 2; ++which) {
    const int64_t K = which == 0 ? H : I;
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows}, strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {(cuuint32_t)(QBK / 2), (cuuint32_t)QBM};
    CUresult r = enc(reinterpret_cast<CUtensorMap *>(which == 0 ? map_xq : map_hq), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                     const_cast<void *>(which == 0 ? xq : hq), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return (int)r;
  }
  for (int which = 0; which < 2; ++which) {
    const bool down = which == 1;
    const int64_t K = down ? I : H, rows_w = down ? H : 2 * I;
    cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)rows_w, (cuuint64_t)S};
    cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)slot_stride};
    cuuint32_t box[3] = {(cuuint32_t)(QBK / 2), (cuuint32_t)(down ? QBN : QBN / 2), 1};
    CUresult r = enc(reinterpret_cast<CUtensorMap *>(down ? map_d : map_gu), CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                     const_cast<uint8_t *>(slots) + (down ? L.d_codes : L.gu_codes), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return (int)r;
    cuuint64_t sdims[3] = {(cuuint64_t)(K / 16), (cuuint64_t)rows_w, (cuuint64_t)S};
    cuuint64_t sstrides[2] = {(cuuint64_t)(K / 16), (cuuint64_t)slot_stride};
    cuuint32_t sbox[3] = {16, (cuuint32_t)(down ? QBN : QBN / 2), 1};
    r = enc(reinterpret_cast<CUtensorMap *>(down ? map_d_sf : map_gu_sf), CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
            const_cast<uint8_t *>(slots) + (down ? L.d_sf : L.gu_sf), sdims, sstrides, sbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return (int)r;
  }
  return 0;
}

// Block-scaled FP4 tensor-core rate: one CTA per SM, `iters` groups of 4 MMAs
// (M = 128, N = n_tile, K = 64) each.  Returns the milliseconds of the launch
// (CUDA events on `s`), or a negative value on error.
double fp4_peak_ms(int n_tile, int iters, int *err, cudaStream_t s) {
  const int sms = tc_num_sms();
  const int smem = Q_A + 256 * 128 + 2 * Q_SF + 64 + 1024;
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return -1.0;
  cudaError_t e;
  if (n_tile == 256) {
    cudaFuncSetAttribute(fp4_peak_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEventRecord(e0, s);
    fp4_peak_kernel<256><<<sms, 128, smem, s>>>(iters, err);
  } else {
    cudaFuncSetAttribute(fp4_peak_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEventRecord(e0, s);
    fp4_peak_kernel<128><<<sms, 128, smem, s>>>(iters, err);
  }
  e = cudaGetLastError();
  cudaEventRecord(e1, s);
  float ms = -1.0f;
  if (e == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess) cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return e == cudaSuccess ? ms : -1.0;
}

}  // namespace ftmoe
