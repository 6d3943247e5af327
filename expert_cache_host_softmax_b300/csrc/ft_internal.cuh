// ft_internal.cuh -- shared declarations of the sm_103a MoE-offload library.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "../../include/ft_moe.h"

namespace ftmoe {

enum { FMT_BF16 = 0, FMT_NVFP4 = 1, FMT_MXFP4 = 2, FMT_FP8 = 3 };
enum { MODE_LRU = 0, MODE_STREAM = 1 };

constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;
constexpr int kMissScaleArgs = 64;   // misses whose global scales travel as kernel arguments
constexpr int kRouteThreads = 1024;       // single-CTA routing / plan kernels
constexpr int kChunkTokens = 32;          // tokens per CTA in the multi-CTA routing path
constexpr int kSmallRoutePairs = 2048;    // calls with T*k up to this route in one CTA

// Byte offsets of the sections of one expert blob (see include/ft_moe.h).
struct BlobLayout {
  int64_t gu_codes, gu_sf, d_codes, d_sf, gscale, bytes;
};

__host__ __device__ inline BlobLayout blob_layout(int fmt, int64_t H, int64_t I) {
  const int64_t HI = H * I;
  BlobLayout b{};
  if (fmt == FMT_BF16) {
    b.gu_codes = 0; b.gu_sf = 0; b.d_codes = 4 * HI; b.d_sf = 0; b.gscale = -1; b.bytes = 6 * HI;
  } else if (fmt == FMT_NVFP4) {
    b.gu_codes = 0; b.gu_sf = HI; b.d_codes = HI + HI / 8; b.d_sf = b.d_codes + HI / 2;
    b.gscale = b.d_sf + HI / 16; b.bytes = b.gscale + 16;
  } else if (fmt == FMT_FP8) {
    // codes, then one fp32 scale per row
    b.gu_codes = 0; b.gu_sf = 2 * HI; b.d_codes = 2 * HI + 8 * I; b.d_sf = b.d_codes + HI;
    b.gscale = -1; b.bytes = b.d_sf + 4 * H;
  } else {
    b.gu_codes = 0; b.gu_sf = HI; b.d_codes = HI + HI / 16; b.d_sf = b.d_codes + HI / 2;
    b.gscale = -1; b.bytes = b.d_sf + HI / 32;
  }
  return b;
}

// Device buffers describing one call's routing and cache plan.
struct PlanBufs {
  int32_t *topk_idx;   // [T*k]
  float *gates;        // [T*k]
  int32_t *offsets;    // [E+1]
  int32_t *perm;       // [T*k]
  int32_t *inv;        // [T*k]
  int32_t *u_expert;   // [Umax]  distinct experts, ascending
  int32_t *u_slot;     // [Umax]
  int32_t *u_hit;      // [Umax]
  int32_t *u_evicted;  // [Umax]
  int4 *u_info;        // [Umax]  {expert, slot, first permuted position, (tokens << 1) | hit}, hits first
  int2 *miss;          // [Umax]  {key, slot} of each miss, ascending expert id (count: n[2])
  int32_t *n;          // [4]: n_unique, n_hit, n_miss, n_evicted
};

// Cache tables (device).
struct CacheBufs {
  int32_t *key_slot;        // [L*E]  slot of key, -1 if not resident
  int32_t *slot_key;        // [S]    key in slot, -1 if free
  const int32_t *order_in;  // [S]    slots, least recent first (free slots first, by index)
  int32_t *order_out;       // [S]
  unsigned long long *stats;  // [16]: cumulative {lookups,hits,misses,evictions,bytes} at 0..4, last call at 8..12
};

struct RouteArgs {
  const float *logits;
  int T, E, k, layer, mode, S;
  int bank_slot0;           // STREAM mode: first slot of the bank that holds this layer
  long long blob_bytes;
  PlanBufs plan;
  CacheBufs cache;
  int32_t *mirror;          // mapped host memory: [0]=seq [1]=n_miss [2..2+Umax) keys [..) slots; may be null
  int umax;
  uint32_t seq;
  // multi-CTA path scratch
  int32_t *chunk_counts;    // [n_chunks][E]
  int32_t *chunk_base;      // [n_chunks][E]
  int n_chunks;
  int pdl;                  // single-CTA route kernel launched with programmatic dependent launch
};

// Launchers (route.cu)
cudaError_t launch_route(const RouteArgs &a, cudaStream_t s);
int route_kernel_count(int T, int k);
cudaError_t launch_topk_only(const float *logits, int T, int E, int k, int32_t *idx, float *gates,
                             cudaStream_t s);
cudaError_t launch_permute_only(const int32_t *idx, int T, int k, int E, int32_t *offsets,
                                int32_t *perm, int32_t *inv, int32_t *chunk_counts,
                                int32_t *chunk_base, cudaStream_t s);
size_t permute_scratch_ints(int T, int k, int E);
void route_init_attributes();

// Expert FFN (ffn_gemv.cu)
// Misses copied on the device: byte ranges of every miss's blob (seg[r] =
// [begin, end), 16-byte aligned; empty ranges allowed) from its pinned host
// blob (device-visible address pool_dev[key]) into its slot.  Ranges 0-1 hold
// what the gate/up projection reads (its rows and scales, and the NVFP4
// global scales at the blob's end), range 2 the down rows and scales.
struct MissCopyArgs {
  const int2 *miss;          // plan.miss
  const int32_t *n;          // plan counts: n[2] = misses
  const uint64_t *pool_dev;
  uint8_t *slots;
  long long slot_stride;
  long long seg[3][2];
};

struct FfnArgs {
  const uint8_t *slot_bank;
  long long slot_stride;
  int H, I, E, k, fmt;
  const __nv_bfloat16 *x;     // [T][H]
  __nv_bfloat16 *h;           // [T*k][I]   permuted order
  float *y;                   // [T*k][H]   permuted order
  PlanBufs plan;
  int umax;
  int only;                   // 0 all, 1 hits only, 2 misses only
  int max_tokens;             // tokens of the call (no expert sees more)
  int *err;                   // device error word: a bounded wait that gave up records its site
  // misses read from host memory (FT_MISS_PULL): device-visible addresses of
  // the pool's blobs [L*E], the call's layer, and the switch
  const uint64_t *pool_dev;
  int layer;
  int pull;
  int pdl;                    // launch with programmatic dependent launch (follows a kernel directly)
  // misses copied inside the gate/up kernel (GEMV calls with FT_MISS_KERNEL):
  // the first copy_rows rows of its grid copy ranges 0-1 of every miss, raise
  // copy_sync[0] = seq, then copy range 2; the misses' CTAs wait for the flag.
  // The down kernel starts after the whole gate/up grid (and so after range 2).
  MissCopyArgs mc;
  int copy_rows;
  int *copy_sync;             // [0] flag, [1] arrival count, [2] role ticket
  int seq;                    // the flag value this call's miss CTAs wait for
  int seq_raised;             // the value its copying CTAs raise (seq, unless a fault is injected)
  // the misses' slots are written while this grid runs (its own copying
  // CTAs): the GEMV variant that reads weights through L2 (ld.global.cg)
  // instead of the read-only path is launched
  int miss_coherent;
  // tensor-core down projection: with out_acc set, each row's gate-weighted
  // y is added into out_acc[token] (fp32, zeroed before) instead of, or with
  // keep_y as well as, being stored to y
  float *out_acc;             // [T][H]
  int keep_y;
  // tensor-core gate/up with NVFP4 or FP8 experts: x as f16, each token row
  // scaled by a power of two (launch_x_to_f16), and the inverse scales
  const __half *xh;           // [T][H]
  const float *xinv;          // [T]
  // NVFP4 gate/up of misses whose copies are still landing their down part
  // (which holds the global scales): the scales, read by the host from the
  // pool, for each missed expert; n = 0 reads them from the slot
  struct {
    int n;
    int expert[kMissScaleArgs];
    float gate[kMissScaleArgs], up[kMissScaleArgs];
  } ms;
};
// Combine fused into the down GEMV (small calls): out[t] = sum_j gates[t][j] *
// y[inv[t*k+j]], written by the last CTA of each feature tile.  counters: one
// int per tile (combine_tiles(H)), zero between calls.  counters == nullptr
// disables the fusion.
struct CombineArgs {
  const float *gates;
  const int32_t *inv;
  __nv_bfloat16 *out;
  int *counters;
  int T;
  int launches;               // down launches of the call that arrive on the counters (0 counts as 1)
};
int combine_tiles(int H);
int gateup_feature_blocks(int H, int I);   // grid.x of the gate/up GEMV
bool gemv_fuses_combine(int T);
cudaError_t launch_gateup(const FfnArgs &a, cudaStream_t s);
cudaError_t launch_down(const FfnArgs &a, const CombineArgs &cb, cudaStream_t s);
// out = bf16(acc) for n values (multiple of 4).
cudaError_t launch_acc_to_bf16(const float *acc, __nv_bfloat16 *out, int64_t n, cudaStream_t s);
cudaError_t launch_combine(const float *y, const float *gates, const int32_t *inv, int T, int k, int H,
                           __nv_bfloat16 *out, cudaStream_t s);
void ffn_init_attributes();

// Ranges [seg0, seg1) of a.seg, of every miss, by a kernel on stream s.
cudaError_t launch_miss_copy(const MissCopyArgs &a, int seg0, int seg1, cudaStream_t s);
int tc_num_sms();   // SMs of the current device

// Expert FFN on the tensor cores (grouped_gemm.cu)
void gemm_init_attributes();
int make_weight_maps(const uint8_t *slots, int64_t slot_stride, int S, int fmt, int H, int I, void *map_gu,
                     void *map_d);
int make_act_map(const void *base, int64_t rows, int K, void *map);
cudaError_t launch_tc_ffn(const FfnArgs &f, bool down, const void *map_h, const void *map_gu, const void *map_d,
                          int *err, int64_t max_rows, cudaStream_t s);
// x [T][H] bf16 -> xh f16 with each row scaled by a power of two that puts its
// largest magnitude in [2^14, 2^15), and xinv[t] = the inverse scale
cudaError_t launch_x_to_f16(const __nv_bfloat16 *x, int T, int H, __half *xh, float *xinv, cudaStream_t s);
// whether the tensor-core gate/up of this weight format multiplies f16 operands
bool tc_gateup_f16(int fmt);

// FP4 x FP4 variant of the tensor-core FFN (gemm_fp4.cu).  Buffers over
// expert-padded rows (see fp4_padded_rows): x and h as e2m1 codes [rows][K/2],
// their E4M3 block scales as 512-byte atoms (128 rows x 4 blocks), x's fp32
// row scales.
struct Fp4Bufs {
  uint8_t *xq, *xsf;
  float *xg;
  uint8_t *hq, *hsf;
};
void fp4_init_attributes();
int64_t fp4_padded_rows(int64_t rows, int64_t umax);
cudaError_t launch_quant_x(const __nv_bfloat16 *x, const PlanBufs &plan, int T, int k, int H, uint8_t *xq,
                           uint8_t *xsf, float *xg, cudaStream_t s);
cudaError_t launch_tc_ffn_fp4(const FfnArgs &f, bool down, const Fp4Bufs &q, const void *map_a, const void *map_b,
                              const void *map_sfb, int *err, int64_t max_rows, cudaStream_t s);
int make_fp4_maps(const uint8_t *slots, int64_t slot_stride, int S, int H, int I, const void *xq, const void *hq,
                  int64_t rows, void *map_xq, void *map_hq, void *map_gu, void *map_d, void *map_gu_sf,
                  void *map_d_sf);
double fp4_peak_ms(int n_tile, int iters, int *err, cudaStream_t s);

// Programmatic dependent launch.  A kernel launched with `pdl` may start
// while the previous kernel on its stream is still running; it must execute
// pdl_wait() before touching anything that kernel writes (pdl_wait returns
// once it has completed and its memory is visible; without the launch
// attribute it returns at once).  pdl_trigger() lets the next kernel launch;
// every kernel here triggers only after its own pdl_wait, so when kernel n
// starts, kernel n-2 has completed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Decode call as one grid (decode_grid.cu): router, copiers, gate/up and down
// items by arrival ticket.  sync: decode_grid_sync_ints(umax) device ints,
// zero at create and after an error.
bool decode_grid_supported(int T, int k, int H, int I);
int decode_grid_sync_ints(int umax);
cudaError_t launch_decode_grid(const RouteArgs &route, const FfnArgs &ffn, const CombineArgs &cb, int *sync,
                               int n_copy, int seq_raised, bool pdl, cudaStream_t s);

// Fused decode layer (decode_layer.cu): one cooperative kernel per call.
bool mega_supported(int E, int T, int k);
cudaError_t launch_decode_layer(const RouteArgs &route, const FfnArgs &ffn, const CombineArgs &cb, int *sync,
                                bool wait_copies, size_t route_smem, cudaStream_t s);
size_t route_small_smem(int E, int S);

// Sets the message ft_last_error(NULL) returns on this thread.
void set_stateless_error(const std::string &msg);

}  // namespace ftmoe
