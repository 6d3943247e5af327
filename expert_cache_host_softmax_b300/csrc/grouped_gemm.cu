// grouped_gemm.cu -- grouped SwiGLU expert FFN on the 5th-generation tensor
// cores (tcgen05 + TMEM), for calls whose experts see many tokens (prefill).
//
// Per distinct expert u of a call (blob in slot u_slot[u]; its tokens sit at
// permuted positions offsets[e] .. offsets[e+1]):
//   gate/up:  [g | u] = x_rows . W_gu^T (fp32 accumulators in TMEM; row i of
//             the expert's tile is x[perm[i] / k], one row per (token, rank)
//             pair)
//             h = bf16( silu(g) * u )     (epilogue)
//   down:     y = h . W_d^T               (fp32), combined in the epilogue:
//             out_acc[token] += gate * y row  (fp32 atomics)
// The pages say only that cached experts run "at GPU speed" ("Why a Huge MoE
// Model Fits on One Consumer GPU"); SwiGLU and this kernel design are ours.
//
// One persistent CTA per SM walks the call's output tiles.  A tile is 128
// token rows x 256 weight rows (gate/up: 128 gate rows + the 128 matching up
// rows, so the SiLU*mul epilogue sees both halves; down: 256 rows of H).
// K advances in blocks of 64 through a ring of shared-memory stages:
//   - gate/up: two gatherer warps copy the stage's 128 x rows (64 K each)
//     straight from x, by token index, into the 128-byte-swizzled A layout
//     (cp.async, 16 bytes a copy; x is small enough to stay in L2 across the
//     N tiles that reuse it), wait for their own copies and fence them into
//     the async proxy before arriving; down: the producer TMA-loads the A box
//     of h;
//   - one producer thread issues, per stage, the TMA load of the weights
//     (and of the down GEMM's A box): BF16 weights land
//     directly in the swizzled layout; NVFP4 / MXFP4 / FP8 codes land raw in a
//     separate ring, and eight converter warps dequantise them (e2m1 x block
//     scale, or the bare E4M3 value) into the swizzled B tile: to f16 for the
//     gate/up of NVFP4 and FP8 experts (one cvt and one packed multiply a
//     pair, exact; x then comes as f16 rows scaled per token by a power of
//     two, see x_to_f16_kernel), to bf16 otherwise (exact too).  The NVFP4
//     per-matrix global scale, the FP8 per-row scales and the inverse row
//     scales of f16 x are applied to the fp32 accumulator in the epilogue.
//   - one thread issues tcgen05.mma (M=128, N=256, K=16, bf16 or f16 operands
//     -> f32) into one of two TMEM accumulators (2 x 256 columns), so the
//     epilogue of a tile overlaps the MMAs of the next;
//   - four epilogue warps read the accumulator with tcgen05.ld (one TMEM lane
//     = one token row per thread) and write h (bf16), or add the row, times
//     its pair's gate, into the token's fp32 output row (through a per-warp
//     transpose, so each reduction covers 8 rows x 64 contiguous bytes; and
//     store y when asked to keep it).
// Every mbarrier wait is bounded in time.  A wait that runs out records an
// error code, raises the CTA's abort flag, and every role drains its own
// in-flight copies before the CTA frees its TMEM and exits.
#include <cuda.h>

#include <algorithm>

#include "ft_internal.cuh"
#include "tc_ptx.cuh"

namespace ftmoe {

namespace {

using namespace tc;

constexpr int BM = 128;          // token rows per tile (one TMEM lane each)
constexpr int BN = 256;          // weight rows per tile (MMA N)
constexpr int BK = 64;           // K per stage: 128 bytes of bf16 (one swizzle atom)
constexpr int A_STAGE = BM * BK * 2;          // 16 KB
constexpr int B_STAGE = BN * BK * 2;          // 32 KB
constexpr uint32_t kTmemCols = 512;           // two accumulators of BN fp32 columns
constexpr int kMaxU = kMaxExperts;

template <int FMT>
struct Cfg {
  // BF16 weights land in the B tile as they are; the other formats' codes
  // land raw and are converted
  static constexpr bool kConv = FMT != FMT_BF16;
  // code bytes per stage: 64 K of each of the 256 B rows (FP4: 32 bytes a row, FP8: 64)
  static constexpr int kRawRow = FMT == FMT_FP8 ? BK : BK / 2;
  static constexpr int kRawStage = BN * kRawRow;
  // stages of A + (bf16) B; the converted formats also have a ring of raw-code stages
  static constexpr int kNS = kConv ? 3 : 4;
  static constexpr int kNR = kConv ? 4 : 0;
  // warp roles: 0 producer, 1 MMA, 2-3 x gatherers (gate/up; idle in down),
  // 4-7 epilogue, 8-15 converters (converted formats) or 8-11 epilogue (BF16)
  static constexpr int kProdWarp = 0, kMmaWarp = 1, kGatherWarp0 = 2, kEpiWarp0 = 4, kConvWarp0 = 8;
  static constexpr int kGatherThreads = 64;
  static constexpr int kConvThreads = kConv ? 256 : 0;
  // epilogue warps: 8 (two per TMEM lane quarter, each half of a tile's
  // columns) where no converter warps take the registers, else 4
  static constexpr int kEpiW = kConv ? 4 : 8;
  static constexpr int kThreads = kConv ? 512 : 384;
  // FULL arrivals per stage: the producer's expect_tx, plus one per converter
  // thread, plus (gate/up) one per gatherer thread
  __host__ __device__ static constexpr int full_count(bool down) {
    return 1 + kConvThreads + (down ? 0 : kGatherThreads);
  }
  // shared memory: [A x kNS][B x kNS][RAW x kNR] then barriers and tables
  static constexpr int kOffB = kNS * A_STAGE;
  static constexpr int kOffRaw = kOffB + kNS * B_STAGE;
  static constexpr int kOffBar = kOffRaw + kNR * kRawStage;
  // barriers: FULL, EMPTY (kNS each), RAWFULL, RAWEMPTY (kNR each), TFULL x2, TEMPTY x2, DRAIN
  static constexpr int kBars = 2 * kNS + 2 * kNR + 5;
  static constexpr int kOffTab = kOffBar + kBars * 8 + 16;
  // down epilogue: one 32 x 16 fp32 transpose block per epilogue warp (rows padded to 20)
  static constexpr int kOffXp = (kOffTab + 4 * (2 * (kMaxU + 1)) + 64 + 15) / 16 * 16;
  static constexpr int kXpStride = 20;
  static constexpr int kSmem = kOffXp + kEpiW * 32 * kXpStride * 4;
  static constexpr int kSmemAlloc = kSmem + 1024;             // room to align the base to 1024
};

struct GemmArgs {
  const uint8_t *slot_bank;
  long long slot_stride;
  int H, I, k;
  const __nv_bfloat16 *x;   // [T][H]
  __nv_bfloat16 *h;         // [T*k][I]
  float *y;                 // [T*k][H]
  PlanBufs plan;
  int only;                 // 0 all, 1 hits, 2 misses
  long long gscale_off;     // byte offset of the NVFP4 global scales in a blob, else -1
  int *err;                 // device error word (first failure code)
  float *out_acc;           // down: out_acc[token] += gate * y row (fp32 atomics), or null
  int keep_y;               // down with out_acc: store y as well
  const __half *xh;         // f16 gate/up (kF16A): x rows scaled per token, and
  const float *xinv;        // the inverse scales
};

// ------------------------------------------------------------------ instruction descriptor

// Instruction descriptor: kind::f16, A = B = bf16, D = f32, K-major A and B,
// N = BN, M = BM.
// The gate/up of NVFP4 and FP8 experts multiplies f16 operands: their codes
// (times an E4M3 block scale) convert to f16 exactly in one step, and x comes
// as f16 rows scaled by a power of two (launch_x_to_f16).  MXFP4 (E8M0 block
// scales beyond f16's range), BF16 and every down GEMM (A = h) stay bf16.
template <int FMT, bool DOWN>
constexpr bool kF16A = !DOWN && (FMT == FMT_NVFP4 || FMT == FMT_FP8);
// kind::f16 with A = B = f16 (format fields 0), D = f32
constexpr uint32_t kIdescF16 = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

// ------------------------------------------------------------------ tiles

struct TileInfo {
  int u, n, mt;     // distinct expert, N tile, M tile
  int row0, rows;   // first permuted row of the tile, valid rows (<= BM)
  int slot;
};

// v[i] *= scale[i] for 16 consecutive weight rows (FP8 row scales; the same
// 64 bytes for every thread of the warp).
__device__ __forceinline__ void row_scale16(const float *scale, float *v) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 s4 = __ldg(reinterpret_cast<const float4 *>(scale) + i);
    v[4 * i] *= s4.x;
    v[4 * i + 1] *= s4.y;
    v[4 * i + 2] *= s4.z;
    v[4 * i + 3] *= s4.w;
  }
}

// Tile t -> (u, n, m): experts in order, then N tiles, then M tiles (M fastest,
// so the CTAs that share a weight tile run side by side).
__device__ __forceinline__ TileInfo decode_tile(int t, const int *s_start, const int *s_mt, int nU, int NTN,
                                                const GemmArgs &a) {
  int lo = 0, hi = nU;  // last u with s_start[u]*NTN <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_start[mid] * NTN <= t) lo = mid;
    else hi = mid;
  }
  TileInfo ti;
  ti.u = lo;
  const int mt = s_mt[lo];
  const int rem = t - s_start[lo] * NTN;
  ti.n = rem / mt;
  ti.mt = rem - ti.n * mt;
  const int e = a.plan.u_expert[lo];
  const int off = a.plan.offsets[e], cnt = a.plan.offsets[e + 1] - off;
  ti.row0 = off + ti.mt * BM;
  ti.rows = min(BM, cnt - ti.mt * BM);
  ti.slot = a.plan.u_slot[lo];
  return ti;
}

// ------------------------------------------------------------------ kernel

template <int FMT, bool DOWN>
__global__ void __launch_bounds__(Cfg<FMT>::kThreads, 1)
    gemm_kernel(GemmArgs a, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB) {
  using C = Cfg<FMT>;
  constexpr int NS = C::kNS, NR = C::kNR;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  unsigned char *sm = smem_raw + (base - raw_base);
  const uint32_t sA = base, sB = base + C::kOffB, sRaw = base + C::kOffRaw;
  const uint32_t bar0 = base + C::kOffBar;
  auto FULL = [&](int s) { return bar0 + 8u * s; };                    // A (and B) of a stage landed
  auto EMPTY = [&](int s) { return bar0 + 8u * (NS + s); };            // stage consumed by the MMAs
  auto RAWFULL = [&](int r) { return bar0 + 8u * (2 * NS + r); };      // FP4 codes landed
  auto RAWEMPTY = [&](int r) { return bar0 + 8u * (2 * NS + NR + r); };  // FP4 codes converted
  auto TFULL = [&](int b) { return bar0 + 8u * (2 * NS + 2 * NR + b); };
  auto TEMPTY = [&](int b) { return bar0 + 8u * (2 * NS + 2 * NR + 2 + b); };
  const uint32_t DRAIN = bar0 + 8u * (2 * NS + 2 * NR + 4);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + C::kOffBar + C::kBars * 8);
  volatile int *s_abort = reinterpret_cast<volatile int *>(sm + C::kOffBar + C::kBars * 8 + 4);
  int *s_start = reinterpret_cast<int *>(sm + C::kOffTab);
  int *s_mt = s_start + (kMaxU + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = DOWN ? a.I : a.H;
  const int nk = K / BK;
  const int NTN = DOWN ? a.H / BN : a.I / (BN / 2);

  // ---- prologue: barriers, TMEM, tile table
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(FULL(s), C::full_count(DOWN));
      mbar_init(EMPTY(s), 1);
    }
    for (int r = 0; r < NR; ++r) {
      mbar_init(RAWFULL(r), 1);
      mbar_init(RAWEMPTY(r), C::kConvThreads);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(TFULL(b), 1);
      mbar_init(TEMPTY(b), C::kEpiW * 32);
    }
    mbar_init(DRAIN, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == C::kMmaWarp) tmem_alloc(smem_u32(s_tmem), kTmemCols);
  const int nU = a.plan.n[0];
  if (warp == C::kEpiWarp0) {
    // per distinct expert: M tiles (0 when filtered out); exclusive prefix in s_start
    int run = 0;
    for (int u0 = 0; u0 < nU; u0 += 32) {
      const int u = u0 + lane;
      int mt = 0;
      if (u < nU) {
        const int e = a.plan.u_expert[u];
        const int cnt = a.plan.offsets[e + 1] - a.plan.offsets[e];
        const int hit = a.plan.u_hit[u];
        const bool sel = a.only == 0 || (a.only == 1 && hit) || (a.only == 2 && !hit);
        mt = sel ? (cnt + BM - 1) / BM : 0;
        s_mt[u] = mt;
      }
      int x = mt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (u < nU) s_start[u] = run + x - mt;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s_start[nU] = run;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int n_tiles = s_start[nU] * NTN;

  if (warp == C::kProdWarp) {
    // ================================================================ producer
    // Per stage: wait for the slot; one expect_tx for the stage's TMA bytes;
    // for down, the A box (128 permuted h rows x 64 K; the gate/up A rows come
    // from the gatherers); for BF16, the two halves of the weight tile; for
    // FP4, the raw codes into their own ring.
    if (lane == 0) {
      int j = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, s_start, s_mt, nU, NTN, a);
        const int r0 = DOWN ? ti.n * BN : ti.n * (BN / 2);            // first weight row (gate rows for gate/up)
        const int r1 = DOWN ? ti.n * BN + BN / 2 : a.I + ti.n * (BN / 2);  // second half (up rows)
        for (int kb = 0; kb < nk; ++kb, ++j) {
          const int s = j % NS;
          if (!mbar_wait(EMPTY(s), ((j / NS) & 1) ^ 1, s_abort, a.err, 10)) { ok = false; break; }
          constexpr uint32_t tx = (DOWN ? A_STAGE : 0) + (C::kConv ? 0 : B_STAGE);
          if constexpr (tx > 0) mbar_arrive_expect_tx(FULL(s), tx);
          else mbar_arrive(FULL(s));
          if constexpr (DOWN) tma_load_2d(sA + s * A_STAGE, &tmA, FULL(s), kb * BK, ti.row0);
          if constexpr (!C::kConv) {
            const uint32_t dst = sB + s * B_STAGE;
            tma_load_3d(dst, &tmB, FULL(s), kb * BK, r0, ti.slot);
            tma_load_3d(dst + B_STAGE / 2, &tmB, FULL(s), kb * BK, r1, ti.slot);
          } else {
            const int rs = j % NR;
            if (!mbar_wait(RAWEMPTY(rs), ((j / NR) & 1) ^ 1, s_abort, a.err, 11)) { ok = false; ++j; break; }
            fence_proxy_async();   // the converters' reads of this slot precede the TMA's writes
            mbar_arrive_expect_tx(RAWFULL(rs), C::kRawStage);
            const uint32_t dst = sRaw + rs * C::kRawStage;
            tma_load_3d(dst, &tmB, RAWFULL(rs), kb * C::kRawRow, r0, ti.slot);
            tma_load_3d(dst + C::kRawStage / 2, &tmB, RAWFULL(rs), kb * C::kRawRow, r1, ti.slot);
          }
        }
      }
      // every TMA this CTA issued must land before the CTA exits
      for (int jj = max(0, j - NS); jj < j; ++jj) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(FULL(jj % NS), (jj / NS) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
      if constexpr (C::kConv) {
        for (int jj = max(0, j - NR); jj < j; ++jj) {
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(RAWFULL(jj % NR), (jj / NR) & 1) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (!DOWN && warp >= C::kGatherWarp0 && warp < C::kGatherWarp0 + C::kGatherThreads / 32) {
    // ================================================================ x gatherers
    // The gate/up A tile holds the x rows of the tile's permuted pairs
    // (token perm[row] / k), copied 16 bytes at a time into the swizzled
    // stage (chunk c of row r at c ^ (r & 7)).  Eight consecutive lanes copy
    // one 128-byte row segment, so a warp's copy reads 4 whole lines of x and
    // fills 512 contiguous bytes of the stage; thread (w, l) copies chunk
    // l & 7 of rows 8 i + 4 w + (l >> 3), i = 0..15.  Rows past the expert's
    // last pair repeat its last row (their results are dropped).  Stages are
    // published LAG stages late: once a later stage's copies are issued, the
    // thread waits for its own copies of the oldest unpublished stage, makes
    // them visible to the tensor core's proxy and arrives on FULL; a tile's
    // stages are all published before the next tile's token indices are
    // loaded.  Deadlock-free for LAG < NS: the stage a gatherer waits to
    // refill was published LAG - 1 or more iterations earlier.
    constexpr int LAG = NS >= 4 ? 2 : 1;
    const int t = tid - C::kGatherWarp0 * 32;
    const int rsub = 4 * (t >> 5) + (lane >> 3), c = lane & 7;
    const uint32_t dsub = rsub * 128 + ((c ^ (rsub & 7)) << 4);
    int j = 0, p0 = 0, np = 0;   // stages p0 .. p0 + np - 1 issued, not yet published
    bool ok = true;
    auto publish_all = [&]() {
      cp_async_wait<0>();
      fence_proxy_async();
      for (; np > 0; --np, ++p0) mbar_arrive(FULL(p0 % NS));
    };
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      if (np > 0) publish_all();
      const TileInfo ti = decode_tile(tile, s_start, s_mt, nU, NTN, a);
      const int last = ti.row0 + ti.rows - 1;
      int tok[BM / 8];
#pragma unroll
      for (int i = 0; i < BM / 8; ++i) tok[i] = a.plan.perm[min(ti.row0 + 8 * i + rsub, last)] / a.k;
      const uint16_t *xsrc = kF16A<FMT, DOWN> ? reinterpret_cast<const uint16_t *>(a.xh)
                                               : reinterpret_cast<const uint16_t *>(a.x);
      const uint16_t *xc = xsrc + c * 8;
      for (int kb = 0; kb < nk; ++kb, ++j) {
        const int s = j % NS;
        if (!mbar_wait(EMPTY(s), ((j / NS) & 1) ^ 1, s_abort, a.err, 14)) { ok = false; break; }
        const uint32_t d = sA + s * A_STAGE + dsub;
#pragma unroll
        for (int i = 0; i < BM / 8; ++i) cp_async16(d + i * 1024, xc + (size_t)tok[i] * a.H + kb * BK);
        cp_async_commit();
        if (np == 0) p0 = j;
        if (++np > LAG) {
          cp_async_wait<LAG>();
          fence_proxy_async();
          mbar_arrive(FULL(p0 % NS));
          ++p0;
          --np;
        }
      }
    }
    // the stages still unpublished; every copy lands before the thread exits
    publish_all();
  } else if (FMT == FMT_FP8 && warp >= C::kConvWarp0) {
    // ================================================================ FP8 converters
    // Each thread expands one B row per stage, 64 E4M3 codes, into the
    // swizzled bf16 tile (chunk c of row t at c ^ (t & 7)); the row scales
    // wait for the epilogue.  Thread t reads its four 16-byte code groups in
    // the order g = sigma(a) ^ i (a = (t >> 1) & 3, sigma = 0 2 3 1): within
    // each 8 lanes both the loads (rows 64 bytes apart) and the swizzled
    // stores then touch 8 distinct 16-byte bank groups.
    const int t = tid - C::kConvWarp0 * 32;
    const uint32_t sig = (0x1320u >> (4 * ((t >> 1) & 3))) & 3u;
    int j = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      for (int kb = 0; kb < nk; ++kb, ++j) {
        const int s = j % NS;
        if (!mbar_wait(EMPTY(s), ((j / NS) & 1) ^ 1, s_abort, a.err, 12)) { ok = false; break; }
        const int rs = j % NR;
        if (!mbar_wait(RAWFULL(rs), (j / NR) & 1, s_abort, a.err, 13)) { ok = false; break; }
        const uint32_t raw = sRaw + rs * C::kRawStage + t * C::kRawRow;
        const uint32_t bdst = sB + s * B_STAGE + t * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t g = sig ^ (uint32_t)i;
          uint4 q;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
                       : "r"(raw + g * 16)
                       : "memory");
          const uint4 v0 = kF16A<FMT, DOWN> ? dequant8_e4m3_f16(q.x, q.y) : dequant8_e4m3(q.x, q.y);
          const uint4 v1 = kF16A<FMT, DOWN> ? dequant8_e4m3_f16(q.z, q.w) : dequant8_e4m3(q.z, q.w);
          const uint32_t d0 = bdst + (((2 * g) ^ (t & 7)) << 4), d1 = bdst + (((2 * g + 1) ^ (t & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d0), "r"(v0.x), "r"(v0.y), "r"(v0.z),
                       "r"(v0.w)
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d1), "r"(v1.x), "r"(v1.y), "r"(v1.z),
                       "r"(v1.w)
                       : "memory");
        }
        mbar_arrive(RAWEMPTY(rs));
        fence_proxy_async();   // this thread's B row is visible to the tensor core's reads
        mbar_arrive(FULL(s));
      }
    }
  } else if (C::kConv && warp >= C::kConvWarp0) {
    // ================================================================ FP4 converters
    // Each thread dequantises one B row per stage from the raw codes into the
    // swizzled bf16 tile (chunk c of row t at c ^ (t & 7)).
    const int t = tid - C::kConvWarp0 * 32;
    const BlobLayout L = blob_layout(FMT, a.H, a.I);
    uint4 sc_cur = make_uint4(0, 0, 0, 0), sc_nxt = make_uint4(0, 0, 0, 0);
    int j = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, s_start, s_mt, nU, NTN, a);
      // this thread's B row in the blob (gate/up: 128 gate rows, then the 128 matching up rows)
      const int brow =
          DOWN ? ti.n * BN + t : (t < BN / 2 ? ti.n * (BN / 2) + t : a.I + ti.n * (BN / 2) + (t - BN / 2));
      const int sf_per_row = K / (FMT == FMT_NVFP4 ? 16 : 32);
      const uint8_t *sf_row = a.slot_bank + (size_t)ti.slot * a.slot_stride + (DOWN ? L.d_sf : L.gu_sf) +
                              (size_t)brow * sf_per_row;
      for (int kb = 0; kb < nk; ++kb, ++j) {
        const int s = j % NS;
        // block scales of the 4 stages of group kb/4 (NVFP4: 16 bytes, MXFP4:
        // 8 bytes), loaded one group ahead
        constexpr int per = FMT == FMT_NVFP4 ? 4 : 2;   // scale bytes per stage
        auto load_group = [&](int g) -> uint4 {
          if (FMT == FMT_NVFP4) return __ldg(reinterpret_cast<const uint4 *>(sf_row + g * 4 * per));
          const uint2 v = __ldg(reinterpret_cast<const uint2 *>(sf_row + g * 4 * per));
          return make_uint4(v.x, v.y, 0, 0);
        };
        if (kb == 0) sc_nxt = load_group(0);
        if ((kb & 3) == 0) {
          sc_cur = sc_nxt;
          if (kb + 4 < nk) sc_nxt = load_group(kb / 4 + 1);
        }
        const int sub = kb & 3;
        float sc[4];
        uint32_t sch[4];   // f16 path: the scales as f16x2 pairs
        if constexpr (FMT == FMT_NVFP4) {
          const uint32_t word = sub == 0 ? sc_cur.x : sub == 1 ? sc_cur.y : sub == 2 ? sc_cur.z : sc_cur.w;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if constexpr (kF16A<FMT, DOWN>) sch[i] = e4m3_to_half2x(word >> (8 * i));
            else sc[i] = e4m3_to_float((word >> (8 * i)) & 0xFFu);
          }
        } else {
          const uint32_t word = (sub >> 1) == 0 ? sc_cur.x : sc_cur.y;
          const uint32_t pair = (word >> (16 * (sub & 1))) & 0xFFFFu;
          sc[0] = sc[1] = e8m0_to_float(pair & 0xFFu);
          sc[2] = sc[3] = e8m0_to_float(pair >> 8);
        }
        // the B slot is free once the MMAs of stage j - NS are done
        if (!mbar_wait(EMPTY(s), ((j / NS) & 1) ^ 1, s_abort, a.err, 12)) { ok = false; break; }
        const int rs = j % NR;
        if (!mbar_wait(RAWFULL(rs), (j / NR) & 1, s_abort, a.err, 13)) { ok = false; break; }
        // rows are 32 bytes apart: lanes 4-7 of every 8 read their second half
        // first, so that each load instruction touches all 32 banks
        const uint32_t raw = sRaw + rs * C::kRawStage + t * 32;
        const uint32_t hsw = ((t >> 2) & 1) * 16;
        uint4 qa, qb;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(qa.x), "=r"(qa.y), "=r"(qa.z), "=r"(qa.w)
                     : "r"(raw + hsw)
                     : "memory");
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(qb.x), "=r"(qb.y), "=r"(qb.z), "=r"(qb.w)
                     : "r"(raw + (hsw ^ 16))
                     : "memory");
        const uint4 q0 = hsw ? qb : qa, q1 = hsw ? qa : qb;
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint32_t bdst = sB + s * B_STAGE + t * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = kF16A<FMT, DOWN> ? dequant8_f16(w[c], sch[c >> 1]) : dequant8(w[c], sc[c >> 1]);
          const uint32_t d = bdst + ((c ^ (t & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                       : "memory");
        }
        // the raw codes have been consumed (the stores above depend on them):
        // the producer may refill this raw slot
        mbar_arrive(RAWEMPTY(rs));
        fence_proxy_async();   // this thread's B row is visible to the tensor core's reads
        mbar_arrive(FULL(s));
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      int j = 0, tl = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tl) {
        const int b = tl & 1;
        if (!mbar_wait(TEMPTY(b), ((tl >> 1) & 1) ^ 1, s_abort, a.err, 20)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + b * BN;
        for (int kb = 0; kb < nk; ++kb, ++j) {
          const int s = j % NS;
          if (!mbar_wait(FULL(s), (j / NS) & 1, s_abort, a.err, 21)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sA + s * A_STAGE, b0 = sB + s * B_STAGE;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16(d, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32),
                     kF16A<FMT, DOWN> ? kIdescF16 : kIdesc, (kb | kk) != 0);
          mma_commit(EMPTY(s));
        }
        if (ok) mma_commit(TFULL(b));
      }
      // every MMA issued must complete before TMEM is freed
      mma_commit(DRAIN);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(DRAIN, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else if (warp >= C::kEpiWarp0 && warp < C::kEpiWarp0 + C::kEpiW) {
    // ================================================================ epilogue
    const int q = warp & 3;            // TMEM lane quarter
    const int row = q * 32 + lane;     // tile row of this thread
    constexpr int NG = C::kEpiW / 4;   // warps per lane quarter, each 1/NG of the columns
    const int grp = (warp - C::kEpiWarp0) >> 2;
    int tl = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tl) {
      const int b = tl & 1;
      const TileInfo ti = decode_tile(tile, s_start, s_mt, nU, NTN, a);
      if (!mbar_wait(TFULL(b), (tl >> 1) & 1, s_abort, a.err, 30)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN;
      float g0 = 1.0f, g1 = 1.0f;
      if (a.gscale_off >= 0) {
        const float *gs = reinterpret_cast<const float *>(a.slot_bank + (size_t)ti.slot * a.slot_stride +
                                                         a.gscale_off);
        g0 = DOWN ? gs[2] : gs[0];
        g1 = gs[1];
      }
      // FP8: the fp32 scales of the tile's weight rows (gate/up: the 128 gate
      // rows and the 128 matching up rows; down: 256 rows of H)
      const float *rs0 = nullptr, *rs1 = nullptr;
      if constexpr (FMT == FMT_FP8) {
        const BlobLayout L = blob_layout(FMT_FP8, a.H, a.I);
        const float *sf = reinterpret_cast<const float *>(a.slot_bank + (size_t)ti.slot * a.slot_stride +
                                                         (DOWN ? L.d_sf : L.gu_sf));
        rs0 = DOWN ? sf + ti.n * BN : sf + ti.n * (BN / 2);
        rs1 = DOWN ? nullptr : sf + a.I + ti.n * (BN / 2);
      }
      const bool valid = row < ti.rows;
      if constexpr (kF16A<FMT, DOWN>) {
        // the row's x came scaled by a power of two: its inverse joins the weights' scales
        const float inv = valid ? a.xinv[a.plan.perm[ti.row0 + row] / a.k] : 1.0f;
        g0 *= inv;
        g1 *= inv;
      }
      if constexpr (!DOWN) {
        __nv_bfloat16 *dst = a.h + (size_t)(ti.row0 + row) * a.I + ti.n * (BN / 2);
#pragma unroll 1
        for (int c = grp * (BN / 2 / NG); c < (grp + 1) * (BN / 2 / NG); c += 16) {
          float gv[16], uv[16];
          tmem_ld16(tb + c, gv);
          tmem_ld16(tb + BN / 2 + c, uv);
          if constexpr (FMT == FMT_FP8) {
            row_scale16(rs0 + c, gv);
            row_scale16(rs1 + c, uv);
          }
          if (valid) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float h2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float g = gv[2 * i + e] * g0, u = uv[2 * i + e] * g1;
                h2[e] = g / (1.0f + expf(-g)) * u;
              }
              pk[i] = pack_bf16x2(h2[0], h2[1]);
            }
            uint4 *o = reinterpret_cast<uint4 *>(dst + c);
            o[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            o[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else {
        float *dst = a.y + (size_t)(ti.row0 + row) * a.H + ti.n * BN;
        // the combine, fused: this row is pair (token t, rank j); its y row,
        // times the pair's gate, goes straight into t's fp32 output row
        float *acc = nullptr;
        float gw = 0.0f;
        if (a.out_acc != nullptr && valid) {
          const int pair = a.plan.perm[ti.row0 + row];
          acc = a.out_acc + (size_t)(pair / a.k) * a.H + ti.n * BN;
          gw = a.plan.gates[pair] * g0;
        }
        const bool store_y = a.out_acc == nullptr || a.keep_y;
        const uint64_t opol = l2_evict_last();   // the output rows stay in L2 for the other pairs' updates
        // The reductions go through a per-warp transpose: lane l holds 16
        // columns of its own row; after the transpose each reduction
        // instruction j covers rows 8 j .. 8 j + 7 of the warp, four lanes a
        // row (64 contiguous bytes), so a warp's instruction touches 8 output
        // rows instead of 32.  Lane l then serves row 8 j + (l >> 2), float4
        // (l & 3) of the 16 columns; that row's output pointer and gate come
        // from its owner lane.
        float *xp =
            reinterpret_cast<float *>(sm + C::kOffXp) + (size_t)((warp - C::kEpiWarp0) * 32) * C::kXpStride;
        float *racc[4];
        float rgw[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int src = 8 * jj + (lane >> 2);
          racc[jj] = reinterpret_cast<float *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(acc), src));
          rgw[jj] = __shfl_sync(0xffffffffu, gw, src);
        }
#pragma unroll 1
        for (int c = grp * (BN / NG); c < (grp + 1) * (BN / NG); c += 16) {
          float v[16];
          tmem_ld16(tb + c, v);
          if constexpr (FMT == FMT_FP8) row_scale16(rs0 + c, v);
          if (valid && store_y) {
            float4 *o = reinterpret_cast<float4 *>(dst + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              o[i] = make_float4(v[4 * i] * g0, v[4 * i + 1] * g0, v[4 * i + 2] * g0, v[4 * i + 3] * g0);
          }
          if (a.out_acc != nullptr) {
            float4 *w4 = reinterpret_cast<float4 *>(xp + lane * C::kXpStride);
#pragma unroll
            for (int i = 0; i < 4; ++i) w4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int r = 8 * jj + (lane >> 2), f4 = lane & 3;
              const float4 t = *reinterpret_cast<const float4 *>(xp + r * C::kXpStride + 4 * f4);
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
  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kMmaWarp) tmem_dealloc(tmem_base, kTmemCols);
}

// ------------------------------------------------------------------ host side

template <int FMT, bool DOWN>
void set_attr() {
  cudaFuncSetAttribute(gemm_kernel<FMT, DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<FMT>::kSmemAlloc);
}

template <int FMT, bool DOWN>
cudaError_t launch(const GemmArgs &a, const CUtensorMap &mapA, const CUtensorMap &mapB, int grid, cudaStream_t s) {
  gemm_kernel<FMT, DOWN><<<grid, Cfg<FMT>::kThreads, Cfg<FMT>::kSmemAlloc, s>>>(a, mapA, mapB);
  return cudaGetLastError();
}

// One token row per CTA: x (bf16) -> f16 scaled by 2^k, k putting the row's
// largest magnitude in [2^14, 2^15) (every element down to 2^-31 of it
// converts exactly), xinv[t] = 2^-k.  A row whose largest magnitude is zero
// or not finite is not scaled.
__global__ void __launch_bounds__(256) x_to_f16_kernel(const __nv_bfloat16 *__restrict__ x, int H,
                                                       __half *__restrict__ xh, float *__restrict__ xinv) {
  __shared__ uint32_t s_wmax[8];
  const int t = blockIdx.x;
  const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
  uint4 *dst = reinterpret_cast<uint4 *>(xh + (size_t)t * H);
  const int nv = H / 8;
  uint32_t m = 0;   // largest |x| as fp32 bits
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const uint4 q = __ldg(src + v);
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
  const float sc = __uint_as_float((uint32_t)(127 + k) << 23);
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const uint4 q = __ldg(src + v);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h2 =
          __floats2half2_rn(__uint_as_float(w[j] << 16) * sc, __uint_as_float(w[j] & 0xFFFF0000u) * sc);
      o[j] = *reinterpret_cast<const uint32_t *>(&h2);
    }
    dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) xinv[t] = __uint_as_float((uint32_t)(127 - k) << 23);
}

}  // namespace

bool tc_gateup_f16(int fmt) { return fmt == FMT_NVFP4 || fmt == FMT_FP8; }

cudaError_t launch_x_to_f16(const __nv_bfloat16 *x, int T, int H, __half *xh, float *xinv, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  x_to_f16_kernel<<<T, 256, 0, s>>>(x, H, xh, xinv);
  return cudaGetLastError();
}

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

static_assert(Cfg<FMT_BF16>::kSmemAlloc <= 227 * 1024, "bf16 smem");
static_assert(Cfg<FMT_NVFP4>::kSmemAlloc <= 227 * 1024, "fp4 smem");
static_assert(Cfg<FMT_FP8>::kSmemAlloc <= 227 * 1024, "fp8 smem");
static_assert(Cfg<FMT_NVFP4>::kThreads == 512 && Cfg<FMT_BF16>::kThreads == 384, "warp roles");
static_assert(Cfg<FMT_BF16>::kGatherThreads == 64 && BM == 128 && BK == 64, "gatherer row map: 2 warps, 8 lanes a row");

int tc_num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

void gemm_init_attributes() {
  set_attr<FMT_BF16, false>();
  set_attr<FMT_BF16, true>();
  set_attr<FMT_NVFP4, false>();
  set_attr<FMT_NVFP4, true>();
  set_attr<FMT_MXFP4, false>();
  set_attr<FMT_MXFP4, true>();
  set_attr<FMT_FP8, false>();
  set_attr<FMT_FP8, true>();
}

// Tensor map over the bf16 activation matrix h [rows][K]: box of 64 K x 128
// rows with the 128-byte swizzle.
int make_act_map(const void *base, int64_t rows, int K, void *map) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return -1;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows}, strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {BK, BM}, estr[2] = {1, 1};
  CUresult r = enc(reinterpret_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                   dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)r;
}

// Tensor maps over the slot bank: 3-D (K, rows, slot).  BF16: box 64 x 128
// elements with the 128-byte swizzle.  FP4: raw code bytes, box 32 x 128.
// FP8: raw code bytes, box 64 x 128.
int make_weight_maps(const uint8_t *slots, int64_t slot_stride, int S, int fmt, int H, int I, void *map_gu,
                     void *map_d) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return -1;
  const BlobLayout L = blob_layout(fmt, H, I);
  for (int which = 0; which < 2; ++which) {
    const bool down = which == 1;
    const int64_t K = down ? I : H, rows = down ? H : 2 * I;
    CUtensorMap *m = reinterpret_cast<CUtensorMap *>(down ? map_d : map_gu);
    void *gaddr = const_cast<uint8_t *>(slots) + (down ? L.d_codes : L.gu_codes);
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    CUtensorMapDataType dt;
    CUtensorMapSwizzle sw;
    if (fmt == FMT_BF16) {
      dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      dims[0] = K; strides[0] = K * 2;
      box[0] = BK;
      sw = CU_TENSOR_MAP_SWIZZLE_128B;
    } else if (fmt == FMT_FP8) {
      dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
      dims[0] = K; strides[0] = K;
      box[0] = BK;
      sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    } else {
      dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
      dims[0] = K / 2; strides[0] = K / 2;
      box[0] = BK / 2;
      sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    }
    dims[1] = rows; dims[2] = S;
    strides[1] = slot_stride;
    box[1] = BN / 2; box[2] = 1;
    CUresult r = enc(m, dt, 3, gaddr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return (int)r;
  }
  return 0;
}

// Grouped gate/up (down=false) or down (down=true) FFN of the call's experts on
// the tensor cores.  map_h: the activation map (make_act_map) over h, the
// down GEMM's A (the gate/up GEMM gathers its x rows itself); map_gu /
// map_d: the slot-bank weight maps.
cudaError_t launch_tc_ffn(const FfnArgs &f, bool down, const void *map_h, const void *map_gu, const void *map_d,
                          int *err, int64_t max_rows, cudaStream_t s) {
  GemmArgs a{};
  a.slot_bank = f.slot_bank;
  a.slot_stride = f.slot_stride;
  a.H = f.H; a.I = f.I; a.k = f.k;
  a.x = f.x; a.h = f.h; a.y = f.y;
  a.plan = f.plan;
  a.only = f.only;
  a.gscale_off = f.fmt == FMT_NVFP4 ? blob_layout(FMT_NVFP4, f.H, f.I).gscale : -1;
  a.err = err;
  a.out_acc = down ? f.out_acc : nullptr;
  a.keep_y = f.keep_y;
  a.xh = f.xh;
  a.xinv = f.xinv;
  const int NTN = down ? f.H / BN : f.I / (BN / 2);
  // M tiles <= ceil(rows / BM) + distinct experts
  const int64_t mtiles = (max_rows + BM - 1) / BM + f.umax;
  const int grid = (int)std::min<int64_t>(tc_num_sms(), std::max<int64_t>(1, mtiles * NTN));
  const CUtensorMap &mA = *reinterpret_cast<const CUtensorMap *>(map_h);   // unused by gate/up
  const CUtensorMap &mB = *reinterpret_cast<const CUtensorMap *>(down ? map_d : map_gu);
  switch (f.fmt) {
    case FMT_BF16: return down ? launch<FMT_BF16, true>(a, mA, mB, grid, s) : launch<FMT_BF16, false>(a, mA, mB, grid, s);
    case FMT_NVFP4:
      return down ? launch<FMT_NVFP4, true>(a, mA, mB, grid, s) : launch<FMT_NVFP4, false>(a, mA, mB, grid, s);
    case FMT_FP8: return down ? launch<FMT_FP8, true>(a, mA, mB, grid, s) : launch<FMT_FP8, false>(a, mA, mB, grid, s);
    default: return down ? launch<FMT_MXFP4, true>(a, mA, mB, grid, s) : launch<FMT_MXFP4, false>(a, mA, mB, grid, s);
  }
}

}  // namespace ftmoe
