/*
 * ft_moe.h -- C ABI of the host-resident-expert MoE layer for B300 (sm_103a).
 *
 * One Mixture-of-Experts layer forward.  The full expert pool sits in pinned
 * host RAM.  A fixed number of GPU expert slots act as one least-recently-used
 * cache, shared by all layers.  Sources:
 *   "FreeToken: Run Frontier MoE Models on Your Own GPU, and the RAM It Takes"
 *   (devpik.com):
 *     section "Why a Huge MoE Model Fits on One Consumer GPU" -- the router
 *       sends each token to a few experts.  The GPU keeps an LRU cache of
 *       expert slots.  A cached expert runs at GPU speed; a miss is streamed
 *       over PCIe.  One global LRU pool is shared across layers.
 *     section "The Real Requirement Is System RAM" -- NVFP4 is 4-bit values
 *       plus an 8-bit scale for every 16 weights.
 *     section "Long Prompts Are the Bottleneck" -- prefill copies all experts
 *       of a layer for each chunk.  The copy of layer N+1 overlaps the compute
 *       of layer N, and the cache must hold the two staging layers.
 *   "FreeToken: Run a 290B MoE Model on One Gaming GPU" (wpnews.pro), section
 *     "VRAM Is Not the Bottleneck You Think It Is" -- the complete pool lives in
 *     system RAM, and VRAM is an LRU cache of recently activated experts.
 *
 * Conventions.
 *   - Every call returns an ft_status code.  On error it changes no state that
 *     a later call depends on, except where a call's own text says otherwise.
 *     ft_last_error() gives a one-line reason.
 *   - "device" pointers are CUDA device memory of the handle's device;
 *     "host" pointers are CPU memory.  The caller owns all pointers it passes.
 *     The library owns every device buffer it allocates, and frees it in
 *     ft_moe_destroy.
 *   - stream arguments are cudaStream_t values passed as void* (0 = legacy
 *     default stream).
 *   - Calls on one handle are not thread-safe; serialise them.
 *   - Layouts are row-major.  bf16 is stored as uint16 bit patterns.
 *
 * Expert blob (the unit the pool holds and a slot caches).  Per expert there
 * are three matrices: gate [I][H], up [I][H] and down [H][I], with K
 * contiguous.  Gate and up are stacked as W_gu [2I][H].
 *   FT_FMT_BF16 : W_gu bf16[2I][H] | W_d bf16[H][I]                (6HI bytes)
 *   FT_FMT_NVFP4: gu codes u8[2I][H/2] | gu scales e4m3[2I][H/16]
 *               | d codes u8[H][I/2]   | d scales e4m3[H][I/16]
 *               | f32 global scale {gate, up, down, 0}          (27HI/16 + 16)
 *   FT_FMT_MXFP4: gu codes u8[2I][H/2] | gu scales e8m0[2I][H/32]
 *               | d codes u8[H][I/2]   | d scales e8m0[H][I/32]         (51HI/32)
 *   FT_FMT_FP8  : gu codes e4m3[2I][H] | gu scales f32[2I]
 *               | d codes e4m3[H][I]   | d scales f32[H]          (3HI + 8I + 4H)
 * FP4 code bytes hold element 2j in the low nibble and 2j+1 in the high
 * nibble.  An NVFP4 weight is e2m1(code) * e4m3(block scale) * global scale.
 * An MXFP4 weight is e2m1(code) * 2^(e8m0 - 127) (OCP Microscaling v1.0).
 * An FP8 weight is e4m3(code) (OCP "FN") * the fp32 scale of its row.  FP8
 * experts are not pulled (FT_MISS_PULL copies them instead).
 */
#ifndef FT_MOE_H_
#define FT_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ft_moe ft_moe; /* opaque handle: slot bank, cache tables, streams, events */

enum ft_fmt { FT_FMT_BF16 = 0, FT_FMT_NVFP4 = 1, FT_FMT_MXFP4 = 2, FT_FMT_FP8 = 3 };

enum ft_mode {
  FT_MODE_LRU = 0,    /* decode: per-call slot lookup, LRU update, miss streaming */
  FT_MODE_STREAM = 1  /* prefill: whole layers streamed into two slot banks (double buffer) */
};

enum ft_status {
  FT_OK = 0,
  FT_ERR_ARG = -1,             /* an argument is out of range or a pointer is NULL */
  FT_ERR_CUDA = -2,            /* a CUDA runtime call failed */
  FT_ERR_OOM = -3,             /* device or pinned allocation failed */
  FT_ERR_NOT_PINNED = -4,      /* a pool pointer is not page-locked host memory */
  FT_ERR_CACHE_TOO_SMALL = -5, /* too few slots for one call (LRU) or two staging layers (STREAM) */
  FT_ERR_STATE = -6,           /* call not valid in the handle's state */
  FT_ERR_TIMEOUT = -7,         /* a bounded host wait for the device expired */
  FT_ERR_DEVICE = -8           /* a kernel reported an error word */
};

/* Cache counters.  A lookup is one distinct (layer, expert) of a forward call;
 * in LRU mode hits + misses = lookups (STREAM-mode lookups are neither).
 * evictions counts misses that displaced a resident expert.  warm_loads counts
 * experts copied by load_pool/reset.  streamed counts experts that STREAM-mode
 * layer staging copied from host memory, hit_d2d those it copied from a cache
 * slot on the device (ft_moe_set_prefill_hit_d2d).  bytes_h2d counts all
 * expert bytes copied host->device. */
typedef struct {
  uint64_t lookups, hits, misses, evictions, warm_loads, streamed, bytes_h2d, hit_d2d;
} ft_stats;

/* Packed bytes of one expert blob in weight_fmt (layouts above), or -1 for a
 * bad format or shape. */
int64_t ft_moe_blob_bytes(int weight_fmt, int hidden, int inter);

/* Creates a layer stack of n_layers MoE layers that share one slot cache.
 *   hidden H, inter I: multiples of 256; n_experts E in 1..512; top_k in
 *   1..min(E, 32); weight_fmt an ft_fmt; n_slots S in 1..65536; max_tokens >= 1
 *   bounds n_tokens of every forward.
 * Allocates on the current CUDA device: S slots of ft_moe_blob_bytes each
 * (rounded up to 256 B), the cache tables, and scratch sized by max_tokens.
 * Errors: FT_ERR_ARG (shape), FT_ERR_CACHE_TOO_SMALL when
 * S < min(E, max_tokens*top_k) (the distinct experts of one call must fit, so
 * a call never evicts one of its own experts), FT_ERR_OOM, FT_ERR_CUDA.
 * *out is set only on FT_OK.
 * Env FT_FAULT=alloc makes it return FT_ERR_OOM before touching the device
 * (host-side fault injection for tests). */
int ft_moe_create(int hidden, int n_experts, int top_k, int inter, int weight_fmt,
                  int n_slots, int n_layers, int max_tokens, ft_moe **out);

/* Registers the host expert pool: host_experts[layer * E + e] points to the
 * blob of expert e of that layer, in page-locked host memory
 * (cudaHostAlloc/cudaHostRegister).  The pointers are not copied.  The memory
 * must outlive the handle.  A contiguous pool is the case
 * ptr[i] = base + i * blob_bytes.  Then warm-fills the cache: keys
 * 0..min(S, L*E)-1 go to slots 0.., with slot 0 the least recently used.
 * Synchronous.  Errors: FT_ERR_ARG (NULL), FT_ERR_NOT_PINNED, FT_ERR_CUDA.
 * Env FT_FAULT=pin returns FT_ERR_NOT_PINNED before touching the device. */
int ft_moe_load_pool(ft_moe *h, const void *const *host_experts);

/* Selects FT_MODE_LRU or FT_MODE_STREAM.  STREAM needs S >= 2*E, room for
 * the two staging layers ("Long Prompts Are the Bottleneck"); the banks are
 * the last 2E slots (bank b = slots S-2E+b*E ..), and the first S-2E slots
 * stay the LRU cache's.  FT_ERR_CACHE_TOO_SMALL otherwise.
 * With prefill hit-D2D off (the default) the call resets the cache and the
 * counters to the mode's initial state (LRU: warm fill; STREAM: an empty
 * cache and both banks empty).  With it on, the cache survives the switch
 * and the counters carry on: entering STREAM mode the cache keeps its most
 * recent S-2E experts, a kept expert at slot >= S-2E moving to the lowest
 * free slot below (least recent first, copied on the device); leaving it, the
 * cache grows back to S slots, its experts where they are and the bank slots
 * free; selecting the current mode again changes nothing.  Synchronous.
 * Errors: FT_ERR_ARG (NULL, bad mode), FT_ERR_CACHE_TOO_SMALL, FT_ERR_DEVICE
 * (a kernel of an earlier call gave up a bounded wait), FT_ERR_CUDA; after
 * FT_ERR_CUDA the cache state is undefined until ft_cache_reset. */
int ft_moe_set_mode(ft_moe *h, int mode);

/* Prefill hit-D2D ("Long Prompts Are the Bottleneck": prefill can skip the
 * experts already in the GPU cache, so that only the others cross PCIe).  on
 * = 1: STREAM-mode staging copies each expert that the cache holds from its
 * slot on the device (counted in hit_d2d, not streamed or bytes_h2d), and
 * ft_moe_set_mode keeps the cache across switches (above).  STREAM mode
 * reads the cache but changes neither its experts nor their recency.  on = 0
 * (default): every staged expert comes from host memory.  Takes effect at the
 * next staging or switch.  Errors: FT_ERR_ARG (NULL, on not 0/1). */
int ft_moe_set_prefill_hit_d2d(ft_moe *h, int on);

/* 1 if prefill hit-D2D is on, 0 if off, FT_ERR_ARG for NULL. */
int ft_moe_prefill_hit_d2d(ft_moe *h);

/* One MoE layer forward for n_tokens tokens (0 <= n_tokens <= max_tokens):
 *   x             device bf16 [n_tokens][H]
 *   router_logits device f32  [n_tokens][E]
 *   out           device bf16 [n_tokens][H]   (written; may not alias x)
 * x and router_logits may not alias the previous call's out either: this
 * call's kernels read them before the previous call's last kernel has
 * completed (they must be final when this call is issued on `stream`, as any
 * input written by earlier work on the stream is).
 * For each token, experts = the top_k largest logits (ties to the lower id),
 * gates = softmax over those top_k logits, and
 * out = sum_j gate_j * W_d (silu(W_g x) * (W_u x)) over the token's experts,
 * with h rounded to bf16 and fp32 accumulation.
 * LRU mode: the distinct experts of the call are looked up in the slot
 * table.  Hits move to MRU in ascending expert id.  Then misses, in ascending
 * id, take the lowest free slot or evict the LRU expert.  All of this is
 * decided on the GPU.  How a miss's blob reaches its slot is set by
 * ft_moe_set_miss_path.  With FT_MISS_COPY the host issues cudaMemcpyAsync on
 * the handle's copy streams, overlapping the FFN of the hits, and the call
 * blocks the host until the GPU's miss list is known: a bounded wait,
 * FT_ERR_TIMEOUT after FT_WAIT_TIMEOUT_MS (default 20000); such a call cannot
 * run under stream capture (FT_ERR_STATE).  With FT_MISS_KERNEL (or
 * FT_MISS_PULL on a GEMV call) the GPU fetches the misses itself: no host
 * wait, and the call can be captured in a CUDA graph (not while profiling).
 * Each launch of such a graph is one more call: it advances the cache state.
 * After a captured call, the synchronising calls (ft_cache_stats and others)
 * wait for the whole device.
 * STREAM mode: bank (layer mod 2) receives all E experts of `layer` before
 * its FFN.  The copy of the next layer starts in this call and overlaps this
 * layer's compute.  With prefill hit-D2D on, the experts that the cache holds
 * are copied from their slots, the others from host memory.
 * Work is ordered after earlier work on `stream`.  out is ready when `stream`
 * reaches the end of this call's work.  Errors: FT_ERR_ARG, FT_ERR_STATE (no
 * pool loaded), FT_ERR_TIMEOUT, FT_ERR_CUDA.  After FT_ERR_TIMEOUT or
 * FT_ERR_CUDA the cache state is undefined until ft_cache_reset. */
int ft_moe_forward(ft_moe *h, int layer, int n_tokens, const void *x,
                   const float *router_logits, void *out, void *stream);

/* Cumulative counters since the last reset/mode change, and those of the
 * last forward call.  Waits for the handle's outstanding work.  Either
 * pointer may be NULL. */
int ft_cache_stats(ft_moe *h, ft_stats *cumulative, ft_stats *last_call);

/* Changes the number of expert slots at run time, returning VRAM to (or
 * taking it from) other users without reloading the pool ("Why a Huge MoE
 * Model Fits on One Consumer GPU": VRAM moves between the expert cache and the
 * KV cache at run time, without a restart).  LRU mode: the cache keeps its
 * most recently used experts, as many as fit, in the same recency order; a
 * kept expert keeps its slot if that slot still exists, else it moves to the
 * lowest free slot (least recent first); new slots start free.  The experts
 * that leave are not counted as evictions of a call; the counters are kept.
 * STREAM mode: the cache (the slots below the banks) follows the same rules
 * onto its new share, n_slots - 2E, and the banks start empty.  The slot bank is reallocated
 * at the new size (old and new coexist during the call) and the kept experts
 * are copied on the device.  CUDA graphs captured from this handle before the
 * call hold the old bank's address and must not be launched after it
 * (capture again).  Waits for the handle's work.  Errors: FT_ERR_ARG,
 * FT_ERR_CACHE_TOO_SMALL (the rules of ft_moe_create / ft_moe_set_mode),
 * FT_ERR_OOM (the handle is unchanged), FT_ERR_CUDA. */
int ft_moe_resize_slots(ft_moe *h, int n_slots);

/* Restores the initial cache state and clears the counters.  LRU mode:
 * warm != 0 warm-fills as load_pool does, warm == 0 leaves every slot free.
 * STREAM mode: an empty cache and both staging banks empty.  Synchronous. */
int ft_cache_reset(ft_moe *h, int warm);

/* The last forward call's cache plan, one entry per distinct expert in
 * ascending id: experts[i], slots[i], hit[i] (1/0), evicted[i] (the displaced
 * key layer*E+e, or -1).  Writes min(count, cap) entries into host arrays
 * (any may be NULL) and sets *n = count.  Waits for the handle's work. */
int ft_cache_trace(ft_moe *h, int32_t *experts, int32_t *slots, int32_t *hit,
                   int32_t *evicted, int cap, int *n);

/* The last forward call's routing, copied to host arrays (any may be NULL):
 * topk_idx i32 [T][k], gates f32 [T][k], offsets i32 [E+1] (start of each
 * expert's group in permuted order), perm i32 [T*k] (pair t*k+j in each
 * permuted position: grouped by expert ascending, stable in pair order) and
 * inv i32 [T*k] (permuted position of each pair).  *n_tokens = T.
 * Waits for the handle's work. */
int ft_moe_last_routing(ft_moe *h, int32_t *topk_idx, float *gates, int32_t *offsets,
                        int32_t *perm, int32_t *inv, int *n_tokens);

/* Diagnostics: the last forward call's intermediate activations, copied to
 * host arrays (either may be NULL), in permuted order:
 * h_act bf16 [T*k][I] (silu(gate) * up, rounded to bf16) and y f32 [T*k][H]
 * (the down projection of h_act before the gate-weighted combine).  On
 * tensor-core calls y is written only while activations are kept
 * (ft_moe_set_keep_activations).  Waits for the handle's work. */
int ft_moe_last_activations(ft_moe *h, uint16_t *h_act, float *y);

/* on != 0: tensor-core calls also store y for ft_moe_last_activations.
 * Default off: the tensor-core down GEMM adds each gate-weighted row straight
 * into an fp32 copy of the output (atomic adds, so the order of a token's k
 * terms, and the last bits of out, may differ between runs) and y never
 * reaches memory.  GEMV calls always store y.  Waits for the handle's work.
 * Errors: FT_ERR_ARG. */
int ft_moe_set_keep_activations(ft_moe *h, int on);

/* Step classes timed by the profiling facility. */
enum ft_prof_class {
  FT_PROF_ROUTE = 0,       /* top-k, permute and cache plan kernels */
  FT_PROF_GATEUP_HIT = 1,  /* gate/up FFN over hits (LRU) or over all experts (STREAM) */
  FT_PROF_GATEUP_MISS = 2, /* gate/up FFN over misses (LRU) */
  FT_PROF_DOWN = 3,        /* down FFN */
  FT_PROF_COMBINE = 4,     /* gate-weighted combine */
  FT_PROF_MISS_COPY = 5,   /* the misses' host->device copies of one call (copy stream) */
  FT_PROF_STREAM_COPY = 6, /* one layer's staging copies in STREAM mode (copy stream) */
  FT_PROF_LAYER = 7,       /* a decode call as one kernel (the decode grid, or the fused decode-layer kernel) */
  FT_PROF_CLASSES = 8
};

/* Profiling: while enabled, every forward brackets each step class with CUDA
 * events on the stream that runs it, and waits at its end for them (so the
 * forward becomes host-synchronous).  Enabling or disabling clears the
 * totals.  ft_moe_profile_read returns, per class (first n classes), the
 * summed milliseconds and the number of timed occurrences. */
int ft_moe_set_profiling(ft_moe *h, int enable);
int ft_moe_profile_read(ft_moe *h, double *ms, int64_t *launches, int n);

/* Which kernel computes the expert FFN (gate/up + SiLU*mul, then down). */
enum ft_ffn_kernel {
  FT_FFN_AUTO = 0, /* tensor cores when the call's distinct experts average >= 64 token rows each */
  FT_FFN_GEMV = 1, /* dequant-fused CUDA-core GEMV: streams each weight once per 8 tokens (decode) */
  FT_FFN_TC = 2    /* tcgen05 grouped GEMM: TMA-fed weight tiles, TMEM accumulators (prefill) */
};

/* Selects the FFN kernel for later forward calls (default FT_FFN_AUTO).  Both
 * compute the same function with fp32 accumulation; they differ in the order
 * of the K-dimension sums only.  FT_FFN_TC: 128-row token tiles times 256
 * weight rows; FP4 and FP8 weights are dequantised exactly to bf16 in shared
 * memory (FP8 row scales multiply the fp32 accumulators).
 * Errors: FT_ERR_ARG; FT_ERR_CUDA when the TMA descriptors of the slot bank
 * could not be encoded at create time (then only the GEMV is available). */
int ft_moe_set_ffn_kernel(ft_moe *h, int which);

/* The FFN kernel the last forward call used: FT_FFN_GEMV or FT_FFN_TC
 * (-1 for NULL). */
int ft_moe_last_ffn_kernel(const ft_moe *h);

/* ---- FP4 x FP4 tensor-core FFN ----
 * "FreeToken: Run Frontier MoE Models on Your Own GPU, and the RAM It Takes",
 * section "The Real Requirement Is System RAM": NVFP4 stores 4-bit values
 * with an 8-bit scale for every 16 weights.  The pages say nothing about the
 * precision of the activations.  With FT_ACT_FP4, tensor-core calls (FT_FFN_TC,
 * or AUTO's choice for prefill-sized calls) also quantise the activations to
 * that layout and multiply FP4 x FP4 on the block-scaled tensor cores
 * (tcgen05.mma kind::mxf4nvf4, fp32 accumulation):
 *   x (per token): g = amax(row) / (6 * 448) (1 for an all-zero row);
 *                  scale s_b = E4M3_rn((amax(block of 16) / 6) / g);
 *                  r_b = 1 / (s_b * g), rounded once (0 where s_b * g is 0);
 *                  code q = e2m1_rn(x * r_b);
 *                  the GEMM multiplies its fp32 result by g (and the weights'
 *                  global scales);
 *   h (per row, in the gate/up epilogue, from its fp32 value): the same with
 *                  g = 1, i.e. E4M3 block scales alone -- so h blocks whose
 *                  largest magnitude is below 6 * 2^-6 (about 0.094) get
 *                  subnormal scales and lose precision, and below 6 * 2^-10
 *                  they quantise to zero.
 * Every decision (amax, divisions, roundings: nearest, ties to even,
 * saturating) is taken in IEEE binary32.  GEMV calls (decode) keep bf16
 * activations.  Only NVFP4 weights: FT_ERR_ARG for other formats.  The
 * first FT_ACT_FP4 call allocates 5 device buffers over (max_tokens * top_k
 * + 128 * min(E, max_tokens * top_k)) rows: about 0.6 * hidden + 0.6 * inter
 * bytes per row.  Synchronises the handle.  Errors: FT_ERR_ARG, FT_ERR_OOM,
 * FT_ERR_CUDA, FT_ERR_DEVICE. */
enum ft_act_format { FT_ACT_BF16 = 0, FT_ACT_FP4 = 1 };
int ft_moe_set_act_format(ft_moe *h, int act_fmt);

/* The current activation format (FT_ACT_BF16 or FT_ACT_FP4; -1 for NULL). */
int ft_moe_act_format(const ft_moe *h);

/* The quantised activations of the last forward call, which must have run
 * the FP4 x FP4 FFN (else FT_ERR_STATE), for the T*k (token, rank) pairs in
 * permuted order (position i of ft_moe_last_routing's perm):
 *   x_codes u8 [T*k][hidden/2]  e2m1 codes of x (element 2j in the low nibble of byte j)
 *   x_sf    u8 [T*k][hidden/16] E4M3 block scales of x
 *   x_g     f32 [T*k]           x's row scale g
 *   h_codes u8 [T*k][inter/2], h_sf u8 [T*k][inter/16]  the same for h (no row scale)
 * Any pointer may be NULL.  Host buffers, owned by the caller.  Synchronises
 * the handle.  Errors: FT_ERR_ARG, FT_ERR_STATE, FT_ERR_CUDA, FT_ERR_DEVICE. */
int ft_moe_last_act_fp4(ft_moe *h, uint8_t *x_codes, uint8_t *x_sf, float *x_g, uint8_t *h_codes, uint8_t *h_sf);

/* Measures the block-scaled FP4 tensor-core rate of the current device: one
 * CTA per SM issues `iters` x 4 MMAs (tcgen05.mma kind::mxf4nvf4, M = 128,
 * N = n_tile (128 or 256), K = 64) on operands already in shared memory;
 * *tflops = 2 * 128 * n_tile * 64 * 4 * iters * SMs / (CUDA-event time).
 * Synchronous (default stream).  Errors: FT_ERR_ARG, FT_ERR_OOM, FT_ERR_CUDA,
 * FT_ERR_DEVICE (ft_last_error(NULL) says which). */
int ft_fp4_tensor_peak(int n_tile, int iters, double *tflops);

/* How LRU-mode misses reach their slots. */
enum ft_miss_path {
  FT_MISS_COPY = 0, /* cudaMemcpyAsync on the handle's copy streams, issued by the host once it has
                       read the GPU's miss list; the hits' FFN overlaps the copies.  GEMV calls
                       with up to 64 misses copy the gate/up bytes of every miss first, so that
                       the misses' gate/up overlaps the copies of their down bytes */
  FT_MISS_PULL = 1, /* the FFN kernels read a missed expert's weights straight from pinned host
                       memory over PCIe and write the same bytes into its slot; no host round
                       trip, so forward returns without waiting and can be captured in a CUDA
                       graph.  Applies to calls on the GEMV kernel; tensor-core calls still copy. */
  FT_MISS_KERNEL = 2, /* the GPU copies the misses from pinned host memory into their slots,
                        reading its own miss list: on GEMV calls the first CTAs of the gate/up
                        kernel copy (gate/up bytes first; the misses' CTAs wait for them, the
                        down kernel for the whole grid), on tensor-core calls copy kernels on
                        the copy stream.  No host round trip: forward returns without waiting
                        and can be captured in a CUDA graph.  SM loads reach ~90 % of the copy
                        engine's PCIe rate and share the SMs with the FFN. */
  FT_MISS_AUTO = 3    /* default: FT_MISS_KERNEL for GEMV (decode) calls on experts of at most
                        8 MiB, where the host round trip costs more than the lower rate;
                        FT_MISS_COPY for larger experts and for tensor-core calls */
};

/* Selects the miss path for later forward calls (default FT_MISS_AUTO).  The
 * cache decisions, counters and results are the same on both paths.  Waits for
 * the handle's outstanding work.  Errors: FT_ERR_ARG. */
int ft_moe_set_miss_path(ft_moe *h, int path);

/* The miss path LRU-mode calls on the GEMV (tensor_core = 0) or on the
 * tensor-core FFN (tensor_core != 0) take: FT_MISS_COPY, FT_MISS_PULL or
 * FT_MISS_KERNEL, with FT_MISS_AUTO resolved (-1 for NULL). */
int ft_moe_miss_path(const ft_moe *h, int tensor_core);

/* on != 0: decode calls (LRU mode, GEMV kernel, at most 16 tokens, E <= 256,
 * not under capture) run as one cooperative kernel: routing and the LRU plan,
 * the hits' gate/up, then (once the copy stream has written a flag after the
 * misses' copies) the misses' gate/up, a grid barrier, and the down projection
 * with the combine.  Default off (separate kernels); the results are identical
 * bit for bit.  The fused kernel waits on the copy stream, so tools that
 * serialise all GPU work (profilers) see it wait out its time limit unless the
 * misses are pulled (FT_MISS_PULL).  Waits for the handle's outstanding work.
 * Errors: FT_ERR_ARG. */
int ft_moe_set_decode_fusion(ft_moe *h, int on);

/* Decode calls as one grid (off by default).  An LRU-mode call that runs the
 * GEMV with the misses copied on the GPU (FT_MISS_KERNEL), with at most 32
 * (token, rank) pairs and at most 4 tokens, runs as a single grid whose CTAs
 * take their role by arrival ticket: the router (top-k, permute, LRU plan),
 * then copiers (the misses from pinned host memory into their slots), then the
 * gate/up GEMV items of every distinct expert (hits first), then the down GEMV
 * items with the combine.  Every CTA waits only for CTAs with smaller tickets,
 * so the grid progresses whatever the order of dispatch; each wait is bounded
 * (FT_ERR_DEVICE at the next synchronising call).  The results are those of
 * the separate route, gate/up and down kernels, bit for bit.  Off (the
 * default): those separate kernels, which measure faster on decode-sized
 * calls (the grid's CTAs carry the registers of its largest role, so fewer
 * fit per SM).  Synchronises the handle.  Errors: FT_ERR_ARG, FT_ERR_DEVICE. */
int ft_moe_set_decode_grid(ft_moe *h, int on);

/* Bytes between consecutive slots in the device slot bank. */
int64_t ft_moe_slot_stride(const ft_moe *h);

/* Number of CUDA kernels the handle has launched since creation (-1 for
 * NULL). */
int64_t ft_moe_kernel_launches(const ft_moe *h);

/* One-line reason for the last failure on h.  With h == NULL: the calling
 * thread's last failure of a call that has no handle -- ft_moe_create or a
 * stateless step (ft_topk_softmax, ft_permute, ft_permute_noalloc).  Never
 * NULL. */
const char *ft_last_error(const ft_moe *h);

/* Waits for outstanding work, frees every device and pinned buffer the
 * handle owns, and frees the handle.  NULL is a no-op. */
int ft_moe_destroy(ft_moe *h);

/* ---- stateless steps (device pointers, asynchronous on `stream`) ---- */

/* Router step: for each of T tokens, the top_k largest of E logits (ties to
 * the lower id, descending) into topk_idx i32 [T][k], and their softmax into
 * gates f32 [T][k].  A NaN logit counts as -inf, so a token always gets k
 * distinct experts (the -inf ones lowest id first); the softmax is plain IEEE
 * arithmetic, so a selected +inf or an all -inf selection gives NaN gates.
 * E in 1..512, k in 1..min(E, 32).  Errors: FT_ERR_ARG, FT_ERR_CUDA. */
int ft_topk_softmax(const float *router_logits, int T, int E, int k, int32_t *topk_idx,
                    float *gates, void *stream);

/* Permute step: stable counting sort of the T*k (token, rank) pairs by
 * expert.  Outputs offsets i32 [E+1], perm i32 [T*k] and inv i32 [T*k], as
 * in ft_moe_last_routing.  Ids outside [0, E) are neither counted nor placed
 * (their inv entries are left unwritten and offsets[E] falls short of T*k).  workspace: device scratch of at least
 * ft_permute_workspace_bytes(T, k, E) bytes, owned by the caller, contents
 * ignored on entry.  Errors: FT_ERR_ARG, FT_ERR_CUDA. */
size_t ft_permute_workspace_bytes(int T, int k, int E);
int ft_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *offsets, int32_t *perm,
               int32_t *inv, void *workspace, size_t workspace_bytes, void *stream);

/* ---- permute without allocation ----
 * The pages have no counterpart to this entry point.  It exists for callers
 * that cannot allocate device memory when they run the permute step.  Examples:
 * a serving loop that keeps cudaMalloc/cudaFree off its hot path, because those
 * calls can synchronise the whole device; or a framework whose device memory is
 * all owned by its own pool allocator, with no way to lend scratch to a library.
 *
 * Same inputs, outputs and result as ft_permute, but with no workspace
 * argument.  Its scratch is one file-scope device array of
 * FT_PERMUTE_NOALLOC_MAX_SCRATCH_BYTES bytes.  Every GPU that loads the library
 * holds that array until the process exits.  The call allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).
 *   - Limit: needs 2 * ceil(T/32) * E * 4 bytes of scratch; larger requests
 *     return FT_ERR_ARG (e.g. E = 256 allows T <= 32768).
 *   - The first call made with a given device current looks up the array's
 *     device address (cudaGetSymbolAddress) once for that device.  Make that
 *     first call before any stream capture.  The address is kept for the
 *     process, per device ordinal: it belongs to that device's primary
 *     context and is not looked up again, so after cudaDeviceReset (or under
 *     another context on the same device) this entry point must not be
 *     called.
 *   - Every call shares the one array and overwrites it.  Calls whose work
 *     overlaps on the GPU (other streams, other threads) race on it; serialise
 *     them, e.g. on one stream.  Nothing in the array needs to start at zero:
 *     each call writes every entry before reading it.
 * Errors: FT_ERR_ARG, FT_ERR_CUDA (ft_last_error(NULL) says which). */
#define FT_PERMUTE_NOALLOC_MAX_SCRATCH_BYTES (2u << 20)
int ft_permute_noalloc(const int32_t *topk_idx, int T, int k, int E, int32_t *offsets, int32_t *perm,
                       int32_t *inv, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* FT_MOE_H_ */
