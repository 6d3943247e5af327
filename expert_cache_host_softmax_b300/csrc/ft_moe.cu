// ft_moe.cu -- handle, C ABI and per-call orchestration.
//
// LRU mode, one forward call on the caller's stream.  The route kernel (GPU:
// top-k, gates, permute, slot lookup, LRU update, miss list) runs first; how
// the misses then reach their slots depends on the miss path:
//   FT_MISS_KERNEL (AUTO's choice for GEMV calls on experts <= 8 MiB): the
//     gate/up GEMV grid's first CTAs copy every miss from pinned host memory
//     into its slot, gate/up bytes first; the misses' CTAs wait for them, the
//     down kernel follows the whole grid.  No host step: forward returns at
//     once and can be captured in a CUDA graph.
//   FT_MISS_COPY (AUTO's choice otherwise): the hits' gate/up (and, for GEMV
//     calls, their down projection) start right after route; the host waits
//     (bounded) for the miss list in mapped memory and issues cudaMemcpyAsync
//     per miss on two copy streams ordered after route, so every earlier reader
//     of an evicted slot has finished; the misses' gate/up and down follow
//     their bytes.
//   FT_MISS_PULL: the GEMV kernels read misses straight from host memory.
// The misses' PCIe transfer overlaps the hits' FFN ("Why a Huge MoE Model
// Fits on One Consumer GPU": a cached expert runs at GPU speed; a miss is
// streamed over PCIe).
//
// STREAM mode ("Long Prompts Are the Bottleneck": each MoE layer copies all of
// its experts for a prefill chunk, and the copy of layer N+1 overlaps the
// compute of layer N): bank (layer mod 2) holds the layer's E experts; the
// two banks are the last 2E slots, the slots below them keep the LRU cache.
// Each call also issues the next layer's copies into the other bank, after
// the FFN that last read that bank.  With prefill hit-D2D (same section:
// experts already in the GPU cache need not cross PCIe) the cached experts
// are copied slot -> bank on the device and mode switches keep the cache.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/ft_moe.h"
#include "ft_internal.cuh"

using namespace ftmoe;

constexpr int kProfRing = 64;   // event pairs per profiled step class
// CTAs (of 128 threads) that copy the misses inside the gate/up GEMV kernel:
// four per SM, 8 KB of 16-byte loads in flight each (measured on decode-35B:
// 148 / 296 / 592 / 1184 CTAs -> 53.4 / 53.4 / 52.8 / 52.1 us per miss, the
// last with 4.6 us more per miss-free layer)
constexpr int kCopyCtas = 592;

struct ft_moe {
  int H = 0, E = 0, k = 0, I = 0, fmt = 0, S = 0, L = 0, Tmax = 0, umax = 0, mode = MODE_LRU;
  int64_t blob_bytes = 0, slot_stride = 0;
  int device = 0;
  uint8_t *slots = nullptr;
  int32_t *key_slot = nullptr, *slot_key = nullptr, *order[2] = {nullptr, nullptr};
  int order_cur = 0;
  unsigned long long *stats_dev = nullptr;
  PlanBufs plan{};
  int32_t *chunk_counts = nullptr, *chunk_base = nullptr;
  __nv_bfloat16 *hbuf = nullptr;
  float *ybuf = nullptr;
  float *out_acc = nullptr;          // [Tmax][H] fp32: tensor-core calls add their gate-weighted rows here
  bool keep_y = false;               // ft_moe_set_keep_activations
  int32_t *mirror_host = nullptr, *mirror_dev = nullptr;
  std::vector<const void *> pool;
  bool pool_loaded = false;
  // miss copies alternate between two copy streams, so that one copy's
  // set-up overlaps the previous copy's transfer; copy_stream joins both
  cudaStream_t copy_stream = nullptr, copy_stream2 = nullptr;
  cudaEvent_t ev_route = nullptr, ev_copy = nullptr, ev_copy2 = nullptr, ev_done = nullptr, ev_d2d = nullptr;
  cudaEvent_t ev_bank_ready[2] = {nullptr, nullptr}, ev_bank_free[2] = {nullptr, nullptr};
  int bank_layer[2] = {-1, -1};
  uint32_t seq = 0;
  int last_T = 0;
  bool any_call = false;
  bool last_tc = false;
  bool captured = false;   // a forward was captured into a graph since the last synchronising call
  uint64_t host_warm = 0, host_streamed = 0, host_bytes = 0, host_d2d = 0;
  uint64_t last_streamed = 0, last_stream_bytes = 0, last_d2d = 0;
  // prefill hit-D2D (ft_moe_set_prefill_hit_d2d): STREAM-mode staging copies
  // the experts that the cache holds from their slots; the cache does not
  // change during STREAM mode, so the host keeps its key -> slot map
  bool hit_d2d = false;
  std::vector<int32_t> stream_key_slot;
  // optional per-step timing (ft_moe_set_profiling)
  bool prof = false;
  // a ring of event pairs per class, folded into the totals only when the
  // ring wraps or the totals are read: timing does not stall the host, so the
  // GPU stays ahead of it and a pair spans its kernels, not launch gaps
  cudaEvent_t prof_ev[FT_PROF_CLASSES][kProfRing][2] = {};
  int prof_head[FT_PROF_CLASSES] = {};
  int prof_count[FT_PROF_CLASSES] = {};
  double prof_ms[FT_PROF_CLASSES] = {};
  int64_t prof_launches[FT_PROF_CLASSES] = {};
  int64_t kernel_launches = 0;
  // tensor-core FFN: TMA descriptors over the slot bank, the kernel choice,
  // and a device error word that bounded waits write when they give up
  alignas(64) unsigned char tmap[2][128] = {};     // weights: gate/up, down
  alignas(64) unsigned char amap[128] = {};        // activations: h
  __half *xh = nullptr;                            // x as f16 rows scaled per token [Tmax][H] (f16 gate/up)
  float *xinv = nullptr;                           // their inverse scales [Tmax]
  bool tmaps_ok = false;
  int ffn_kernel = FT_FFN_AUTO;
  int *err_dev = nullptr;
  int *combine_counters = nullptr;   // per feature tile, for the combine fused into the down GEMV
  uint64_t *pool_dev = nullptr;      // device-visible addresses of the pool's blobs [L*E] (FT_MISS_PULL)
  int *mega_sync = nullptr;          // fused decode layer: plan flag, copy flag, grid barrier count and generation
  int *copy_sync = nullptr;          // misses copied inside the gate/up kernel: flag, arrival count, role ticket
  int32_t *seq_ring = nullptr;       // pinned: seq_ring[seq % 64] = seq, the source of the copy-flag write
  bool decode_fused = false;   // ft_moe_set_decode_fusion
  bool decode_grid = false;    // ft_moe_set_decode_grid: eligible decode calls as one grid
  int *grid_sync = nullptr;    // the decode grid's flags and counters
  int miss_path = FT_MISS_AUTO;
  // FP4 x FP4 variant of the tensor-core FFN (ft_moe_set_act_format): buffers
  // over expert-padded rows and their TMA maps (xq, hq, gate/up codes, down codes)
  int act_fmt = FT_ACT_BF16;
  Fp4Bufs q{};
  int64_t q_rows = 0;
  alignas(64) unsigned char qmap[6][128] = {};   // xq, hq, gate/up codes, down codes, their block scales
  bool qmaps_ok = false;
  std::string err;
};

namespace {

thread_local std::string g_create_err;

int fail(ft_moe *h, int code, const std::string &msg) {
  if (h) h->err = msg;
  else g_create_err = msg;
  return code;
}

int cuda_fail(ft_moe *h, cudaError_t e, const char *what) {
  return fail(h, FT_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define FT_CUDA(h, call)                              \
  do {                                                \
    cudaError_t e_ = (call);                          \
    if (e_ != cudaSuccess) return cuda_fail(h, e_, #call); \
  } while (0)

bool fault(const char *what) {
  const char *f = std::getenv("FT_FAULT");
  return f && std::strcmp(f, what) == 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t blob_bytes_of(int fmt, int H, int I) {
  if (fmt < 0 || fmt > 3 || H <= 0 || I <= 0 || H % 256 || I % 256) return -1;
  return blob_layout(fmt, H, I).bytes;
}

template <class T>
cudaError_t dev_alloc(T **p, size_t n) {
  return cudaMalloc(reinterpret_cast<void **>(p), n * sizeof(T) + 16);
}

void free_all(ft_moe *h) {
  cudaFree(h->slots);
  cudaFree(h->key_slot);
  cudaFree(h->slot_key);
  cudaFree(h->order[0]);
  cudaFree(h->order[1]);
  cudaFree(h->stats_dev);
  cudaFree(h->plan.topk_idx);
  cudaFree(h->plan.gates);
  cudaFree(h->plan.offsets);
  cudaFree(h->plan.perm);
  cudaFree(h->plan.inv);
  cudaFree(h->plan.u_expert);
  cudaFree(h->plan.u_slot);
  cudaFree(h->plan.u_hit);
  cudaFree(h->plan.u_evicted);
  cudaFree(h->plan.u_info);
  cudaFree(h->plan.miss);
  cudaFree(h->plan.n);
  cudaFree(h->chunk_counts);
  cudaFree(h->chunk_base);
  cudaFree(h->hbuf);
  cudaFree(h->ybuf);
  cudaFree(h->out_acc);
  cudaFree(h->xh);
  cudaFree(h->xinv);
  cudaFree(h->err_dev);
  cudaFree(h->combine_counters);
  cudaFree(h->pool_dev);
  cudaFree(h->mega_sync);
  cudaFree(h->copy_sync);
  cudaFree(h->grid_sync);
  cudaFree(h->q.xq);
  cudaFree(h->q.xsf);
  cudaFree(h->q.xg);
  cudaFree(h->q.hq);
  cudaFree(h->q.hsf);
  if (h->mirror_host) cudaFreeHost(h->mirror_host);
  if (h->seq_ring) cudaFreeHost(h->seq_ring);
  if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
  if (h->copy_stream2) cudaStreamDestroy(h->copy_stream2);
  for (cudaEvent_t ev : {h->ev_route, h->ev_copy, h->ev_copy2, h->ev_done, h->ev_d2d, h->ev_bank_ready[0], h->ev_bank_ready[1],
                         h->ev_bank_free[0], h->ev_bank_free[1]})
    if (ev) cudaEventDestroy(ev);
  for (auto &cls : h->prof_ev)
    for (auto &pair : cls)
      for (cudaEvent_t ev : pair)
        if (ev) cudaEventDestroy(ev);
}

// Profiling: events around one step class on the stream it runs on.
// Folds the oldest recorded pair of class c into the totals (waits for it).
void prof_fold_oldest(ft_moe *h, int c) {
  const int i = (h->prof_head[c] - h->prof_count[c] + kProfRing) % kProfRing;
  float ms = 0.f;
  if (cudaEventSynchronize(h->prof_ev[c][i][1]) == cudaSuccess &&
      cudaEventElapsedTime(&ms, h->prof_ev[c][i][0], h->prof_ev[c][i][1]) == cudaSuccess) {
    h->prof_ms[c] += ms;
    h->prof_launches[c] += 1;
  }
  --h->prof_count[c];
}
void prof_begin(ft_moe *h, int cls, cudaStream_t s) {
  if (!h->prof) return;
  if (h->prof_count[cls] == kProfRing) prof_fold_oldest(h, cls);
  cudaEventRecord(h->prof_ev[cls][h->prof_head[cls]][0], s);
}
void prof_end(ft_moe *h, int cls, cudaStream_t s) {
  if (!h->prof) return;
  cudaEventRecord(h->prof_ev[cls][h->prof_head[cls]][1], s);
  h->prof_head[cls] = (h->prof_head[cls] + 1) % kProfRing;
  ++h->prof_count[cls];
}
// Folds every recorded pair into the totals (waits for them).
void prof_collect(ft_moe *h) {
  for (int c = 0; c < FT_PROF_CLASSES; ++c)
    while (h->prof_count[c] > 0) prof_fold_oldest(h, c);
}

// Waits for everything the handle has issued, then checks the device error
// word (set by a kernel whose bounded wait gave up).
int sync_handle(ft_moe *h) {
  if (h->captured) {
    FT_CUDA(h, cudaDeviceSynchronize());
    h->captured = false;
  } else if (h->any_call) {
    FT_CUDA(h, cudaEventSynchronize(h->ev_done));
  }
  FT_CUDA(h, cudaStreamSynchronize(h->copy_stream));
  FT_CUDA(h, cudaStreamSynchronize(h->copy_stream2));
  int code = 0;
  FT_CUDA(h, cudaMemcpy(&code, h->err_dev, sizeof code, cudaMemcpyDeviceToHost));
  if (code != 0) {
    FT_CUDA(h, cudaMemset(h->err_dev, 0, sizeof(int)));
    // an aborted kernel may have left its flags or counters mid-way
    FT_CUDA(h, cudaMemset(h->mega_sync, 0, 4 * sizeof(int)));
    FT_CUDA(h, cudaMemset(h->copy_sync, 0, 4 * sizeof(int)));
    FT_CUDA(h, cudaMemset(h->grid_sync, 0, sizeof(int) * decode_grid_sync_ints(h->umax)));
    FT_CUDA(h, cudaMemset(h->combine_counters, 0, sizeof(int) * combine_tiles(h->H)));
    return fail(h, FT_ERR_DEVICE, "a kernel gave up a bounded wait (site " + std::to_string(code) + ")");
  }
  return FT_OK;
}

// Whether this call's FFN runs on the tensor cores: forced by
// ft_moe_set_ffn_kernel, else when the call's experts average at least 64
// token rows each (below that the weight-streaming GEMV wins).
bool use_tc(const ft_moe *h, int T) {
  if (!h->tmaps_ok) return false;
  if (h->ffn_kernel == FT_FFN_GEMV) return false;
  if (h->ffn_kernel == FT_FFN_TC) return true;
  const int64_t rows = (int64_t)T * h->k, distinct = std::min<int64_t>(h->E, rows);
  return rows >= 64 * distinct;
}

cudaError_t run_ffn(ft_moe *h, const FfnArgs &fa, bool down, bool tc, int T, cudaStream_t s,
                    const CombineArgs &cb = CombineArgs{}) {
  if (tc && h->act_fmt == FT_ACT_FP4) {
    if (!down && fa.only != 2) {
      // x quantised once per token into the expert-padded rows (before the first gate/up launch)
      cudaError_t e = launch_quant_x(fa.x, fa.plan, T, h->k, h->H, h->q.xq, h->q.xsf, h->q.xg, s);
      if (e != cudaSuccess) return e;
      h->kernel_launches += 1;
    }
    return launch_tc_ffn_fp4(fa, down, h->q, h->qmap[down ? 1 : 0], h->qmap[down ? 3 : 2], h->qmap[down ? 5 : 4],
                             h->err_dev, (int64_t)T * h->k, s);
  }
  if (tc) {
    FfnArgs f = fa;
    if (!down && tc_gateup_f16(h->fmt)) {
      f.xh = h->xh;
      f.xinv = h->xinv;
      if (fa.only != 2) {
        // x as scaled f16 rows, once per call (before the first gate/up launch)
        cudaError_t e = launch_x_to_f16(fa.x, T, h->H, h->xh, h->xinv, s);
        if (e != cudaSuccess) return e;
        h->kernel_launches += 1;
      }
    }
    return launch_tc_ffn(f, down, h->amap, h->tmap[0], h->tmap[1], h->err_dev, (int64_t)T * h->k, s);
  }
  return down ? launch_down(fa, cb, s) : launch_gateup(fa, s);
}

// Initial cache state of the current mode; clears the counters.
int reset_tables(ft_moe *h, bool warm) {
  FT_CUDA(h, cudaSetDevice(h->device));
  if (int rc = sync_handle(h)) return rc;
  std::vector<int32_t> key_slot((size_t)h->L * h->E, -1), slot_key(h->S, -1), order(h->S);
  int n = 0;
  if (h->mode == MODE_LRU && warm) n = (int)std::min<int64_t>(h->S, (int64_t)h->L * h->E);
  for (int s = 0; s < n; ++s) {
    slot_key[s] = s;
    key_slot[s] = s;
  }
  // free slots first (ascending index), then the warm keys, least recent first
  int pos = 0;
  for (int s = n; s < h->S; ++s) order[pos++] = s;
  for (int s = 0; s < n; ++s) order[pos++] = s;
  FT_CUDA(h, cudaMemcpy(h->key_slot, key_slot.data(), key_slot.size() * 4, cudaMemcpyHostToDevice));
  FT_CUDA(h, cudaMemcpy(h->slot_key, slot_key.data(), slot_key.size() * 4, cudaMemcpyHostToDevice));
  FT_CUDA(h, cudaMemcpy(h->order[0], order.data(), order.size() * 4, cudaMemcpyHostToDevice));
  h->order_cur = 0;
  FT_CUDA(h, cudaMemset(h->stats_dev, 0, 16 * sizeof(unsigned long long)));
  FT_CUDA(h, cudaMemset(h->mega_sync, 0, 4 * sizeof(int)));
  FT_CUDA(h, cudaMemset(h->copy_sync, 0, 4 * sizeof(int)));
  FT_CUDA(h, cudaMemset(h->grid_sync, 0, sizeof(int) * decode_grid_sync_ints(h->umax)));
  FT_CUDA(h, cudaMemset(h->combine_counters, 0, sizeof(int) * combine_tiles(h->H)));
  h->host_warm = h->host_streamed = h->host_bytes = h->host_d2d = 0;
  h->last_streamed = h->last_stream_bytes = h->last_d2d = 0;
  h->bank_layer[0] = h->bank_layer[1] = -1;
  h->stream_key_slot.assign(h->mode == MODE_STREAM ? key_slot.size() : 0, -1);
  h->last_T = 0;
  if (h->pool_loaded) {
    for (int s = 0; s < n; ++s)
      FT_CUDA(h, cudaMemcpyAsync(h->slots + (size_t)s * h->slot_stride, h->pool[s], h->blob_bytes,
                                 cudaMemcpyHostToDevice, h->copy_stream));
    FT_CUDA(h, cudaStreamSynchronize(h->copy_stream));
    h->host_warm = n;
    h->host_bytes = (uint64_t)n * h->blob_bytes;
  }
  return FT_OK;
}

// Slots that belong to the LRU cache in `mode` with S slots: all of them in
// LRU mode; in STREAM mode the last 2E slots are the two staging banks ("Long
// Prompts Are the Bottleneck": the cache must hold the two staging layers).
int cache_slots(const ft_moe *h, int mode, int S) { return mode == MODE_LRU ? S : S - 2 * h->E; }

// First slot of staging bank b (STREAM mode).
int64_t bank_slot0(const ft_moe *h, int b) { return (int64_t)h->S - 2 * h->E + (int64_t)b * h->E; }

// STREAM mode: make bank (layer mod 2) receive all experts of `layer`, after
// the FFN that last read that bank.  With prefill hit-D2D an expert that the
// cache holds is copied from its slot on the device (second copy stream),
// the others from host memory; copy_stream joins both.
int stage_layer(ft_moe *h, int layer) {
  const int b = layer & 1;
  if (h->bank_layer[b] == layer) return FT_OK;
  const int64_t bank0 = bank_slot0(h, b);
  FT_CUDA(h, cudaStreamWaitEvent(h->copy_stream, h->ev_bank_free[b], 0));
  prof_begin(h, FT_PROF_STREAM_COPY, h->copy_stream);
  int n_d2d = 0;
  for (int e = 0; e < h->E; ++e) {
    const size_t key = (size_t)layer * h->E + e;
    uint8_t *dst = h->slots + (size_t)(bank0 + e) * h->slot_stride;
    const int from = h->hit_d2d && key < h->stream_key_slot.size() ? h->stream_key_slot[key] : -1;
    if (from < 0) {
      FT_CUDA(h, cudaMemcpyAsync(dst, h->pool[key], h->blob_bytes, cudaMemcpyHostToDevice, h->copy_stream));
      continue;
    }
    if (n_d2d++ == 0) FT_CUDA(h, cudaStreamWaitEvent(h->copy_stream2, h->ev_bank_free[b], 0));
    FT_CUDA(h, cudaMemcpyAsync(dst, h->slots + (size_t)from * h->slot_stride, h->blob_bytes,
                               cudaMemcpyDeviceToDevice, h->copy_stream2));
  }
  if (n_d2d > 0) {
    FT_CUDA(h, cudaEventRecord(h->ev_d2d, h->copy_stream2));
    FT_CUDA(h, cudaStreamWaitEvent(h->copy_stream, h->ev_d2d, 0));
  }
  prof_end(h, FT_PROF_STREAM_COPY, h->copy_stream);
  FT_CUDA(h, cudaEventRecord(h->ev_bank_ready[b], h->copy_stream));
  h->bank_layer[b] = layer;
  h->last_streamed += h->E - n_d2d;
  h->last_stream_bytes += (uint64_t)(h->E - n_d2d) * h->blob_bytes;
  h->last_d2d += n_d2d;
  return FT_OK;
}

// The cache's keys, least recent first, and its key -> slot table, read from
// the device (the order list holds the free slots in front of the keys).
int read_cache(ft_moe *h, std::vector<int32_t> &key_slot, std::vector<int32_t> &recency) {
  const int S = h->S;
  std::vector<int32_t> slot_key(S), order(S);
  key_slot.resize((size_t)h->L * h->E);
  FT_CUDA(h, cudaMemcpy(slot_key.data(), h->slot_key, sizeof(int32_t) * S, cudaMemcpyDeviceToHost));
  FT_CUDA(h, cudaMemcpy(key_slot.data(), h->key_slot, sizeof(int32_t) * key_slot.size(), cudaMemcpyDeviceToHost));
  FT_CUDA(h, cudaMemcpy(order.data(), h->order[h->order_cur], sizeof(int32_t) * S, cudaMemcpyDeviceToHost));
  recency.clear();
  for (int s : order)
    if (s >= 0 && s < S && slot_key[s] >= 0) recency.push_back(slot_key[s]);
  return FT_OK;
}

// The cache re-planned onto the first n_cache of n_slots slots ("Why a Huge
// MoE Model Fits on One Consumer GPU": VRAM moves between the expert cache
// and other users at run time).  The most recent keys that fit stay, in the
// same recency order; a kept key keeps its slot if it is below n_cache, else
// it takes the lowest free slot (least recent key first).  from[s] is the old
// slot whose bytes slot s must receive (-1: none).  The order list has the
// free slots first, by index, then the keys, least recent first.
struct CachePlan {
  std::vector<int32_t> slot_key, key_slot, order, from;
};

CachePlan plan_cache(const std::vector<int32_t> &key_slot, const std::vector<int32_t> &recency, int n_cache,
                     int n_slots) {
  CachePlan p;
  p.slot_key.assign(n_slots, -1);
  p.key_slot.assign(key_slot.size(), -1);
  p.from.assign(n_slots, -1);
  const size_t n_keep = std::min<size_t>(recency.size(), (size_t)std::max(n_cache, 0));
  const std::vector<int32_t> keep(recency.end() - n_keep, recency.end());
  for (int32_t key : keep) {
    const int s = key_slot[key];
    if (s < n_cache) {
      p.slot_key[s] = key;
      p.key_slot[key] = s;
      p.from[s] = s;
    }
  }
  int next_free = 0;
  for (int32_t key : keep) {
    if (p.key_slot[key] >= 0) continue;
    while (p.slot_key[next_free] >= 0) ++next_free;
    p.slot_key[next_free] = key;
    p.key_slot[key] = next_free;
    p.from[next_free] = key_slot[key];
  }
  for (int s = 0; s < n_slots; ++s)
    if (p.slot_key[s] < 0) p.order.push_back(s);
  for (int32_t key : keep) p.order.push_back(p.key_slot[key]);
  return p;
}

// FT_MISS_AUTO: the device copy (no host round trip, ~10 % lower PCIe rate,
// shares the SMs) for decode calls (GEMV) on small experts, where the round
// trip's ~8 us weighs more; the copy engine (full PCIe rate) for large
// experts and for tensor-core calls, whose own run time hides the round trip
constexpr int64_t kAutoDeviceCopyMaxBytes = 8ll << 20;
int effective_miss_path(const ft_moe *h, bool tc) {
  if (h->miss_path != FT_MISS_AUTO) return h->miss_path;
  return !tc && h->blob_bytes <= kAutoDeviceCopyMaxBytes ? FT_MISS_KERNEL : FT_MISS_COPY;
}

int64_t wait_timeout_ms() {
  const char *v = std::getenv("FT_WAIT_TIMEOUT_MS");
  return v ? std::max<int64_t>(1, std::atoll(v)) : 20000;
}

// Bounded host wait for the route kernel's miss list (mapped host memory).
int wait_plan(ft_moe *h) {
  if (fault("timeout")) return fail(h, FT_ERR_TIMEOUT, "injected wait timeout (FT_FAULT=timeout)");
  const auto t0 = std::chrono::steady_clock::now();
  const int64_t limit = wait_timeout_ms();
  volatile int32_t *flag = h->mirror_host;
  for (uint64_t spin = 0; *flag != (int32_t)h->seq; ++spin) {
    if ((spin & 1023) == 1023) {
      cudaError_t q = cudaEventQuery(h->ev_route);
      if (q != cudaSuccess && q != cudaErrorNotReady) return cuda_fail(h, q, "route kernel");
      if (q == cudaSuccess && *flag != (int32_t)h->seq)
        return fail(h, FT_ERR_DEVICE, "route kernel finished without publishing its miss list");
      const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0).count();
      if (ms > limit) return fail(h, FT_ERR_TIMEOUT, "timed out waiting for the miss list");
    }
    __builtin_ia32_pause();
  }
  std::atomic_thread_fence(std::memory_order_acquire);
  return FT_OK;
}

// Issues the call's miss copies (after the GPU's miss list is known): one
// cudaMemcpyAsync per miss, alternating between the two copy streams, joined
// on copy_stream.  Returns the number of misses, or a negative status.
int issue_miss_copies(ft_moe *h) {
  if (int rc = wait_plan(h)) return rc;
  const int n_miss = h->mirror_host[1];
  if (n_miss <= 0) return 0;
  prof_begin(h, FT_PROF_MISS_COPY, h->copy_stream);
  for (int i = 0; i < n_miss; ++i) {
    const int key = h->mirror_host[2 + i], slot = h->mirror_host[2 + h->umax + i];
    if (key < 0 || key >= h->L * h->E || slot < 0 || slot >= h->S)
      return fail(h, FT_ERR_DEVICE, "miss list entry out of range");
    FT_CUDA(h, cudaMemcpyAsync(h->slots + (size_t)slot * h->slot_stride, h->pool[key], h->blob_bytes,
                               cudaMemcpyHostToDevice, (i & 1) ? h->copy_stream2 : h->copy_stream));
  }
  if (n_miss > 1) {
    FT_CUDA(h, cudaEventRecord(h->ev_copy2, h->copy_stream2));
    FT_CUDA(h, cudaStreamWaitEvent(h->copy_stream, h->ev_copy2, 0));
  }
  prof_end(h, FT_PROF_MISS_COPY, h->copy_stream);
  return n_miss;
}

// A decode call (LRU mode, GEMV, few tokens) as one cooperative kernel: route,
// gate/up of the hits, [the copies land] gate/up of the misses, down and
// combine.  The copy stream tells the kernel that the misses have landed by
// writing the call's sequence number (the mirror's first word) into a device
// flag after the expert copies.
int forward_fused(ft_moe *h, RouteArgs &ra, int layer, int n_tokens, const void *x, void *out, bool pull,
                  cudaStream_t stream) {
  FfnArgs fa{};
  fa.slot_bank = h->slots;
  fa.slot_stride = h->slot_stride;
  fa.H = h->H; fa.I = h->I; fa.E = h->E; fa.k = h->k; fa.fmt = h->fmt;
  fa.x = reinterpret_cast<const __nv_bfloat16 *>(x);
  fa.h = h->hbuf;
  fa.y = h->ybuf;
  fa.plan = h->plan;
  fa.umax = (int)std::min<int64_t>(h->E, (int64_t)n_tokens * h->k);
  fa.max_tokens = n_tokens;
  fa.err = h->err_dev;
  fa.pool_dev = h->pool_dev;
  fa.layer = layer;
  fa.pull = pull ? 1 : 0;
  CombineArgs cb{};
  cb.gates = h->plan.gates;
  cb.inv = h->plan.inv;
  cb.out = reinterpret_cast<__nv_bfloat16 *>(out);
  cb.counters = h->combine_counters;
  cb.T = n_tokens;
  h->last_tc = false;
  // the value the copy stream writes into the kernel's copy flag; a ring, so
  // that a later call cannot overwrite it before the copy engine reads it
  int32_t *release = h->seq_ring + (h->seq % 64);
  *release = (int32_t)h->seq;
  prof_begin(h, FT_PROF_LAYER, stream);
  FT_CUDA(h, launch_decode_layer(ra, fa, cb, h->mega_sync, !pull, route_small_smem(h->E, h->S), stream));
  prof_end(h, FT_PROF_LAYER, stream);
  // the host's wait for the miss list polls this: it completes when the kernel does
  FT_CUDA(h, cudaEventRecord(h->ev_route, stream));
  h->kernel_launches += 1;
  h->order_cur ^= 1;
  if (!pull) {
    const int n_miss = issue_miss_copies(h);
    if (n_miss != 0) {
      // after the copies, or at once if the host side failed: the kernel must
      // not wait out its time limit (its results are then undefined)
      cudaError_t e = cudaMemcpyAsync(h->mega_sync + 1, release, sizeof(int32_t), cudaMemcpyHostToDevice,
                                      h->copy_stream);
      if (n_miss < 0) return n_miss;
      if (e != cudaSuccess) return cuda_fail(h, e, "copy-flag write");
    }
  }
  FT_CUDA(h, cudaEventRecord(h->ev_done, stream));
  return FT_OK;
}

// A decode call (LRU mode, GEMV, misses copied on the GPU, <= 32 pairs) as
// one grid: router, copiers, gate/up and down items by arrival ticket (see
// decode_grid.cu).  No host step; capturable in a CUDA graph.
constexpr int kGridCopyCtas = 296;
int forward_grid(ft_moe *h, RouteArgs &ra, int layer, int n_tokens, const void *x, void *out, bool capturing,
                 cudaStream_t stream) {
  FfnArgs fa{};
  fa.slot_bank = h->slots;
  fa.slot_stride = h->slot_stride;
  fa.H = h->H; fa.I = h->I; fa.E = h->E; fa.k = h->k; fa.fmt = h->fmt;
  fa.x = reinterpret_cast<const __nv_bfloat16 *>(x);
  fa.h = h->hbuf;
  fa.y = h->ybuf;
  fa.plan = h->plan;
  fa.umax = (int)std::min<int64_t>(h->E, (int64_t)n_tokens * h->k);
  fa.max_tokens = n_tokens;
  fa.err = h->err_dev;
  fa.pool_dev = h->pool_dev;
  fa.layer = layer;
  const BlobLayout bl = blob_layout(h->fmt, h->H, h->I);
  MissCopyArgs &mc = fa.mc;
  mc.miss = h->plan.miss;
  mc.n = h->plan.n;
  mc.pool_dev = h->pool_dev;
  mc.slots = h->slots;
  mc.slot_stride = h->slot_stride;
  mc.seg[0][0] = 0;
  mc.seg[0][1] = bl.d_codes;
  mc.seg[1][0] = bl.gscale >= 0 ? bl.gscale : 0;
  mc.seg[1][1] = bl.gscale >= 0 ? h->blob_bytes : 0;
  mc.seg[2][0] = bl.d_codes;
  mc.seg[2][1] = bl.gscale >= 0 ? bl.gscale : h->blob_bytes;
  CombineArgs cb{};
  cb.gates = h->plan.gates;
  cb.inv = h->plan.inv;
  cb.out = reinterpret_cast<__nv_bfloat16 *>(out);
  cb.counters = h->combine_counters;
  cb.T = n_tokens;
  h->last_tc = false;
  // FT_FAULT=devwait: the copy flags are raised with a value nobody waits for
  const int seq_raised = fault("devwait") ? (int)h->seq ^ 0x40000000 : (int)h->seq;
  const bool pdl = !h->prof && !capturing;
  prof_begin(h, FT_PROF_LAYER, stream);
  FT_CUDA(h, launch_decode_grid(ra, fa, cb, h->grid_sync, kGridCopyCtas, seq_raised, pdl, stream));
  prof_end(h, FT_PROF_LAYER, stream);
  h->kernel_launches += 1;
  h->order_cur ^= 1;
  if (capturing) h->captured = true;
  else FT_CUDA(h, cudaEventRecord(h->ev_done, stream));
  return FT_OK;
}

}  // namespace

void ftmoe::set_stateless_error(const std::string &msg) { g_create_err = msg; }

extern "C" {

int64_t ft_moe_blob_bytes(int weight_fmt, int hidden, int inter) { return blob_bytes_of(weight_fmt, hidden, inter); }

int ft_moe_create(int hidden, int n_experts, int top_k, int inter, int weight_fmt, int n_slots, int n_layers,
                  int max_tokens, ft_moe **out) {
  if (!out) return fail(nullptr, FT_ERR_ARG, "out is NULL");
  if (blob_bytes_of(weight_fmt, hidden, inter) < 0 || hidden > 8192 || inter > 8192)
    return fail(nullptr, FT_ERR_ARG, "hidden/inter must be multiples of 256 in 256..8192 and weight_fmt 0..3");
  if (n_experts < 1 || n_experts > kMaxExperts) return fail(nullptr, FT_ERR_ARG, "n_experts must be in 1..512");
  if (top_k < 1 || top_k > std::min(n_experts, kMaxTopK)) return fail(nullptr, FT_ERR_ARG, "top_k must be in 1..min(E,32)");
  if (n_layers < 1 || n_slots < 1 || max_tokens < 1 || n_slots > (1 << 16) ||
      (int64_t)n_layers * n_experts > (1LL << 30) || (int64_t)max_tokens * top_k > (1LL << 30))
    return fail(nullptr, FT_ERR_ARG, "n_layers, max_tokens must be positive; n_slots in 1..65536");
  const int umax = (int)std::min<int64_t>(n_experts, (int64_t)max_tokens * top_k);
  if (n_slots < umax)
    return fail(nullptr, FT_ERR_CACHE_TOO_SMALL,
                "n_slots < min(E, max_tokens*top_k): one call's experts would not fit in the cache");
  if (fault("alloc")) return fail(nullptr, FT_ERR_OOM, "injected allocation failure (FT_FAULT=alloc)");

  ft_moe *h = new ft_moe();
  h->H = hidden; h->E = n_experts; h->k = top_k; h->I = inter; h->fmt = weight_fmt;
  h->S = n_slots; h->L = n_layers; h->Tmax = max_tokens; h->umax = umax;
  h->blob_bytes = blob_bytes_of(weight_fmt, hidden, inter);
  h->slot_stride = (h->blob_bytes + 255) / 256 * 256;
  auto bail = [&](int rc) { free_all(h); delete h; return rc; };
  cudaError_t e = cudaGetDevice(&h->device);
  if (e != cudaSuccess) { cuda_fail(nullptr, e, "cudaGetDevice"); return bail(FT_ERR_CUDA); }
  const size_t TK = (size_t)max_tokens * top_k;
  const size_t chunk_ints = permute_scratch_ints(max_tokens, top_k, n_experts) / 2;
  bool ok = cudaMalloc(&h->slots, (size_t)n_slots * h->slot_stride) == cudaSuccess &&
            dev_alloc(&h->key_slot, (size_t)n_layers * n_experts) == cudaSuccess &&
            dev_alloc(&h->slot_key, n_slots) == cudaSuccess && dev_alloc(&h->order[0], n_slots) == cudaSuccess &&
            dev_alloc(&h->order[1], n_slots) == cudaSuccess && dev_alloc(&h->stats_dev, 16) == cudaSuccess &&
            dev_alloc(&h->plan.topk_idx, TK) == cudaSuccess && dev_alloc(&h->plan.gates, TK) == cudaSuccess &&
            dev_alloc(&h->plan.offsets, n_experts + 1) == cudaSuccess && dev_alloc(&h->plan.perm, TK) == cudaSuccess &&
            dev_alloc(&h->plan.inv, TK) == cudaSuccess && dev_alloc(&h->plan.u_expert, umax) == cudaSuccess &&
            dev_alloc(&h->plan.u_slot, umax) == cudaSuccess && dev_alloc(&h->plan.u_hit, umax) == cudaSuccess &&
            dev_alloc(&h->plan.u_evicted, umax) == cudaSuccess && dev_alloc(&h->plan.n, 4) == cudaSuccess &&
            cudaMalloc(&h->plan.u_info, sizeof(int4) * (size_t)umax) == cudaSuccess &&
            cudaMalloc(&h->plan.miss, sizeof(int2) * (size_t)umax) == cudaSuccess &&
            dev_alloc(&h->chunk_counts, chunk_ints) == cudaSuccess &&
            dev_alloc(&h->chunk_base, chunk_ints) == cudaSuccess &&
            dev_alloc(&h->hbuf, TK * inter) == cudaSuccess && dev_alloc(&h->ybuf, TK * hidden) == cudaSuccess &&
            dev_alloc(&h->out_acc, (size_t)max_tokens * hidden) == cudaSuccess &&
            cudaMalloc(&h->xh, sizeof(__half) * (size_t)max_tokens * hidden) == cudaSuccess &&
            dev_alloc(&h->xinv, (size_t)max_tokens) == cudaSuccess &&
            dev_alloc(&h->err_dev, 4) == cudaSuccess && cudaMemset(h->err_dev, 0, 16) == cudaSuccess &&
            dev_alloc(&h->mega_sync, 4) == cudaSuccess && cudaMemset(h->mega_sync, 0, 16) == cudaSuccess &&
            dev_alloc(&h->copy_sync, 4) == cudaSuccess && cudaMemset(h->copy_sync, 0, 16) == cudaSuccess &&
            dev_alloc(&h->grid_sync, decode_grid_sync_ints(umax)) == cudaSuccess &&
            cudaMemset(h->grid_sync, 0, sizeof(int) * decode_grid_sync_ints(umax)) == cudaSuccess &&
            dev_alloc(&h->combine_counters, combine_tiles(hidden)) == cudaSuccess &&
            cudaMemset(h->combine_counters, 0, sizeof(int) * combine_tiles(hidden)) == cudaSuccess;
  if (!ok) { cudaGetLastError(); fail(nullptr, FT_ERR_OOM, "device allocation failed"); return bail(FT_ERR_OOM); }
  if (cudaHostAlloc(&h->mirror_host, sizeof(int32_t) * (2 + 2 * (size_t)umax), cudaHostAllocMapped) != cudaSuccess ||
      cudaHostGetDevicePointer(reinterpret_cast<void **>(&h->mirror_dev), h->mirror_host, 0) != cudaSuccess) {
    cudaGetLastError();
    fail(nullptr, FT_ERR_OOM, "mapped pinned allocation failed");
    return bail(FT_ERR_OOM);
  }
  std::memset(h->mirror_host, 0, sizeof(int32_t) * (2 + 2 * (size_t)umax));
  if (cudaHostAlloc(&h->seq_ring, sizeof(int32_t) * 64, cudaHostAllocDefault) != cudaSuccess) {
    cudaGetLastError();
    fail(nullptr, FT_ERR_OOM, "pinned allocation failed");
    return bail(FT_ERR_OOM);
  }
  ok = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking) == cudaSuccess &&
       cudaStreamCreateWithFlags(&h->copy_stream2, cudaStreamNonBlocking) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->ev_route, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->ev_copy, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->ev_copy2, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->ev_d2d, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->ev_done, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->ev_bank_ready[0], cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->ev_bank_ready[1], cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->ev_bank_free[0], cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->ev_bank_free[1], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) { cuda_fail(nullptr, cudaGetLastError(), "stream/event creation"); return bail(FT_ERR_CUDA); }
  route_init_attributes();
  ffn_init_attributes();
  gemm_init_attributes();
  fp4_init_attributes();
  // the tensor-core FFN takes BF16, NVFP4 and MXFP4 (FP8 experts run on the GEMV)
  h->tmaps_ok =
                make_weight_maps(h->slots, h->slot_stride, h->S, h->fmt, h->H, h->I, h->tmap[0], h->tmap[1]) == 0 &&
                make_act_map(h->hbuf, (int64_t)TK, h->I, h->amap) == 0;
  if (int rc = reset_tables(h, false)) { g_create_err = h->err; return bail(rc); }
  *out = h;
  return FT_OK;
}

int ft_moe_load_pool(ft_moe *h, const void *const *host_experts) {
  if (!h || !host_experts) return fail(h, FT_ERR_ARG, "NULL handle or pool table");
  if (fault("pin")) return fail(h, FT_ERR_NOT_PINNED, "injected unpinned pool (FT_FAULT=pin)");
  const size_t n = (size_t)h->L * h->E;
  for (size_t i = 0; i < n; ++i) {
    if (!host_experts[i]) return fail(h, FT_ERR_ARG, "NULL expert pointer at " + std::to_string(i));
    cudaPointerAttributes at{};
    cudaError_t e = cudaPointerGetAttributes(&at, host_experts[i]);
    if (e != cudaSuccess || at.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      return fail(h, FT_ERR_NOT_PINNED, "expert " + std::to_string(i) + " is not in page-locked host memory");
    }
  }
  // device-visible address of every blob, for misses read over PCIe by the kernels
  std::vector<uint64_t> dev_ptrs(n);
  for (size_t i = 0; i < n; ++i) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, host_experts[i]) != cudaSuccess || at.devicePointer == nullptr) {
      cudaGetLastError();
      return fail(h, FT_ERR_NOT_PINNED, "expert " + std::to_string(i) + " has no device-visible mapping");
    }
    dev_ptrs[i] = reinterpret_cast<uint64_t>(at.devicePointer);
  }
  FT_CUDA(h, cudaSetDevice(h->device));
  if (!h->pool_dev) FT_CUDA(h, cudaMalloc(&h->pool_dev, n * sizeof(uint64_t)));
  FT_CUDA(h, cudaMemcpy(h->pool_dev, dev_ptrs.data(), n * sizeof(uint64_t), cudaMemcpyHostToDevice));
  h->pool.assign(host_experts, host_experts + n);
  h->pool_loaded = true;
  return reset_tables(h, true);
}

int ft_moe_set_mode(ft_moe *h, int mode) {
  if (!h || (mode != MODE_LRU && mode != MODE_STREAM)) return fail(h, FT_ERR_ARG, "bad mode");
  if (mode == MODE_STREAM && h->S < 2 * h->E)
    return fail(h, FT_ERR_CACHE_TOO_SMALL, "STREAM mode needs n_slots >= 2*E (two staging layers)");
  FT_CUDA(h, cudaSetDevice(h->device));
  if (int rc = sync_handle(h)) return rc;
  if (!h->hit_d2d) {
    h->mode = mode;
    return reset_tables(h, true);
  }
  if (mode == h->mode) return FT_OK;
  // prefill hit-D2D: the cache lives through the switch, shrunk onto the
  // slots below the staging banks (or grown back to all S), in place: the
  // keys that move go from slots >= S - 2E to free slots below it, so no copy
  // reads a slot that another one writes
  std::vector<int32_t> key_slot, recency;
  if (int rc = read_cache(h, key_slot, recency)) return rc;
  const CachePlan p = plan_cache(key_slot, recency, cache_slots(h, mode, h->S), h->S);
  for (int s = 0; s < h->S; ++s)
    if (p.from[s] >= 0 && p.from[s] != s)
      FT_CUDA(h, cudaMemcpyAsync(h->slots + (size_t)s * h->slot_stride, h->slots + (size_t)p.from[s] * h->slot_stride,
                                 h->blob_bytes, cudaMemcpyDeviceToDevice, h->copy_stream));
  FT_CUDA(h, cudaStreamSynchronize(h->copy_stream));
  FT_CUDA(h, cudaMemcpy(h->slot_key, p.slot_key.data(), sizeof(int32_t) * h->S, cudaMemcpyHostToDevice));
  FT_CUDA(h, cudaMemcpy(h->order[0], p.order.data(), sizeof(int32_t) * h->S, cudaMemcpyHostToDevice));
  FT_CUDA(h, cudaMemcpy(h->key_slot, p.key_slot.data(), sizeof(int32_t) * p.key_slot.size(), cudaMemcpyHostToDevice));
  h->order_cur = 0;
  h->mode = mode;
  h->bank_layer[0] = h->bank_layer[1] = -1;
  if (mode == MODE_STREAM) h->stream_key_slot = p.key_slot;
  else h->stream_key_slot.clear();
  return FT_OK;
}

// Changes the slot count ("Why a Huge MoE Model Fits on One Consumer GPU":
// VRAM moves between the expert cache and other users at run time, without a
// restart).  The cache keeps its most recently used keys, as many as fit, in
// the same recency order; a kept key keeps its slot if the slot still exists,
// else takes the lowest free slot (least recent key first); new slots are
// free.  The slot bank is reallocated at the new size and the kept blobs are
// copied into it on the device; nothing is read from host memory.
int ft_moe_resize_slots(ft_moe *h, int n_slots) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (n_slots < 1 || n_slots > (1 << 16)) return fail(h, FT_ERR_ARG, "n_slots must be in 1..65536");
  if (n_slots < h->umax)
    return fail(h, FT_ERR_CACHE_TOO_SMALL, "n_slots < min(E, max_tokens*top_k)");
  if (h->mode == MODE_STREAM && n_slots < 2 * h->E)
    return fail(h, FT_ERR_CACHE_TOO_SMALL, "STREAM mode needs n_slots >= 2*E (two staging layers)");
  FT_CUDA(h, cudaSetDevice(h->device));
  if (int rc = sync_handle(h)) return rc;
  std::vector<int32_t> key_slot, recency;
  if (int rc = read_cache(h, key_slot, recency)) return rc;
  const CachePlan p = plan_cache(key_slot, recency, cache_slots(h, h->mode, n_slots), n_slots);
  // the new bank, the kept blobs copied into it, then the tables
  uint8_t *bank = nullptr;
  int32_t *dslot_key = nullptr, *dorder0 = nullptr, *dorder1 = nullptr;
  if (cudaMalloc(&bank, (size_t)n_slots * h->slot_stride) != cudaSuccess ||
      dev_alloc(&dslot_key, n_slots) != cudaSuccess || dev_alloc(&dorder0, n_slots) != cudaSuccess ||
      dev_alloc(&dorder1, n_slots) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(bank);
    cudaFree(dslot_key);
    cudaFree(dorder0);
    cudaFree(dorder1);
    return fail(h, FT_ERR_OOM, "device allocation for the resized cache failed");
  }
  for (int s = 0; s < n_slots; ++s)
    if (p.from[s] >= 0)
      FT_CUDA(h, cudaMemcpyAsync(bank + (size_t)s * h->slot_stride, h->slots + (size_t)p.from[s] * h->slot_stride,
                                 h->blob_bytes, cudaMemcpyDeviceToDevice, h->copy_stream));
  FT_CUDA(h, cudaStreamSynchronize(h->copy_stream));
  FT_CUDA(h, cudaMemcpy(dslot_key, p.slot_key.data(), sizeof(int32_t) * n_slots, cudaMemcpyHostToDevice));
  FT_CUDA(h, cudaMemcpy(dorder0, p.order.data(), sizeof(int32_t) * n_slots, cudaMemcpyHostToDevice));
  FT_CUDA(h, cudaMemcpy(h->key_slot, p.key_slot.data(), sizeof(int32_t) * p.key_slot.size(), cudaMemcpyHostToDevice));
  cudaFree(h->slots);
  cudaFree(h->slot_key);
  cudaFree(h->order[0]);
  cudaFree(h->order[1]);
  h->slots = bank;
  h->slot_key = dslot_key;
  h->order[0] = dorder0;
  h->order[1] = dorder1;
  h->order_cur = 0;
  h->S = n_slots;
  h->bank_layer[0] = h->bank_layer[1] = -1;
  if (h->mode == MODE_STREAM) h->stream_key_slot = p.key_slot;
  const size_t TK = (size_t)h->Tmax * h->k;
  h->tmaps_ok =
                make_weight_maps(h->slots, h->slot_stride, h->S, h->fmt, h->H, h->I, h->tmap[0], h->tmap[1]) == 0 &&
                make_act_map(h->hbuf, (int64_t)TK, h->I, h->amap) == 0;
  if (h->q.xq)
    h->qmaps_ok = make_fp4_maps(h->slots, h->slot_stride, h->S, h->H, h->I, h->q.xq, h->q.hq, h->q_rows, h->qmap[0],
                                h->qmap[1], h->qmap[2], h->qmap[3], h->qmap[4], h->qmap[5]) == 0;
  if (h->act_fmt == FT_ACT_FP4 && !h->qmaps_ok) h->act_fmt = FT_ACT_BF16;
  return FT_OK;
}

int ft_moe_set_prefill_hit_d2d(ft_moe *h, int on) {
  if (!h || (on != 0 && on != 1)) return fail(h, FT_ERR_ARG, "NULL handle or on not 0/1");
  h->hit_d2d = on != 0;
  return FT_OK;
}

int ft_moe_prefill_hit_d2d(ft_moe *h) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  return h->hit_d2d ? 1 : 0;
}

int ft_cache_reset(ft_moe *h, int warm) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  return reset_tables(h, warm != 0);
}

int ft_moe_forward(ft_moe *h, int layer, int n_tokens, const void *x, const float *router_logits, void *out,
                   void *stream_) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (!h->pool_loaded) return fail(h, FT_ERR_STATE, "no expert pool loaded");
  if (layer < 0 || layer >= h->L) return fail(h, FT_ERR_ARG, "layer out of range");
  if (n_tokens < 0 || n_tokens > h->Tmax) return fail(h, FT_ERR_ARG, "n_tokens out of range");
  h->last_streamed = h->last_stream_bytes = h->last_d2d = 0;
  h->last_T = n_tokens;
  if (n_tokens == 0) return FT_OK;
  if (!x || !router_logits || !out) return fail(h, FT_ERR_ARG, "NULL x, router_logits or out");
  if (!aligned16(x) || !aligned16(router_logits) || !aligned16(out))
    return fail(h, FT_ERR_ARG, "x, router_logits and out must be 16-byte aligned");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  FT_CUDA(h, cudaSetDevice(h->device));
  const bool tc = use_tc(h, n_tokens);
  const int miss_path = effective_miss_path(h, tc);
  // misses read by the kernels over PCIe: no host round trip (GEMV calls only)
  // (FP8 row scales sit outside the chunks the pulling kernels copy: FP8 misses are copied)
  const bool pull = h->mode == MODE_LRU && miss_path == FT_MISS_PULL && !tc && h->fmt != FMT_FP8;
  // misses copied on the device: no host round trip either
  const bool kcopy = h->mode == MODE_LRU && miss_path == FT_MISS_KERNEL;
  cudaStreamCaptureStatus cs;
  FT_CUDA(h, cudaStreamIsCapturing(stream, &cs));
  const bool capturing = cs != cudaStreamCaptureStatusNone;
  if (capturing && (h->mode != MODE_LRU || !(pull || kcopy)))
    return fail(h, FT_ERR_STATE,
                "only LRU-mode forward with FT_MISS_KERNEL (or FT_MISS_PULL on the GEMV) can be captured");
  if (capturing && h->prof) return fail(h, FT_ERR_STATE, "profiling is on: forward cannot be captured");
  const int bank = layer & 1;
  if (h->mode == MODE_STREAM) {
    if (int rc = stage_layer(h, layer)) return rc;
    const int nxt = layer + 1 < h->L ? layer + 1 : 0;
    if ((nxt & 1) != bank)
      if (int rc = stage_layer(h, nxt)) return rc;
    FT_CUDA(h, cudaStreamWaitEvent(stream, h->ev_bank_ready[bank], 0));
  }
  h->any_call = true;
  ++h->seq;
  RouteArgs ra{};
  ra.logits = router_logits;
  ra.T = n_tokens; ra.E = h->E; ra.k = h->k; ra.layer = layer; ra.mode = h->mode; ra.S = h->S;
  ra.bank_slot0 = h->mode == MODE_STREAM ? (int)bank_slot0(h, bank) : 0;
  ra.blob_bytes = h->blob_bytes;
  ra.plan = h->plan;
  ra.cache.key_slot = h->key_slot;
  ra.cache.slot_key = h->slot_key;
  ra.cache.order_in = h->order[h->order_cur];
  ra.cache.order_out = h->order[h->order_cur ^ 1];
  ra.cache.stats = h->stats_dev;
  ra.mirror = (h->mode == MODE_LRU && !pull && !kcopy) ? h->mirror_dev : nullptr;
  ra.umax = h->umax;
  ra.seq = h->seq;
  ra.chunk_counts = h->chunk_counts;
  ra.chunk_base = h->chunk_base;
  // follows the previous call's last kernel directly (STREAM mode waits on a copy event first)
  ra.pdl = h->mode == MODE_LRU && !h->prof && !capturing;
  if (h->decode_fused && h->mode == MODE_LRU && !tc && !kcopy && !capturing && h->fmt != FMT_FP8 &&
      mega_supported(h->E, n_tokens, h->k))
    return forward_fused(h, ra, layer, n_tokens, x, out, pull, stream);
  if (h->decode_grid && kcopy && !tc && gemv_fuses_combine(n_tokens) &&
      decode_grid_supported(n_tokens, h->k, h->H, h->I))
    return forward_grid(h, ra, layer, n_tokens, x, out, capturing, stream);
  prof_begin(h, FT_PROF_ROUTE, stream);
  FT_CUDA(h, launch_route(ra, stream));
  prof_end(h, FT_PROF_ROUTE, stream);
  h->kernel_launches += route_kernel_count(n_tokens, h->k) + 2;  // + gate/up, down (+ combine below)
  if (h->mode == MODE_LRU) h->order_cur ^= 1;
  // the copy stream forks from here (also under capture: the copies join back below)
  if (!capturing || kcopy) FT_CUDA(h, cudaEventRecord(h->ev_route, stream));

  FfnArgs fa{};
  fa.slot_bank = h->slots;
  fa.slot_stride = h->slot_stride;
  fa.H = h->H; fa.I = h->I; fa.E = h->E; fa.k = h->k; fa.fmt = h->fmt;
  fa.x = reinterpret_cast<const __nv_bfloat16 *>(x);
  fa.h = h->hbuf;
  fa.y = h->ybuf;
  fa.plan = h->plan;
  fa.umax = (int)std::min<int64_t>(h->E, (int64_t)n_tokens * h->k);
  fa.max_tokens = n_tokens;
  fa.err = h->err_dev;
  fa.pool_dev = h->pool_dev;
  fa.layer = layer;
  fa.pull = pull ? 1 : 0;
  h->last_tc = tc;
  bool copies_before_down = false;
  // small calls on the GEMV: the combine runs inside the down kernel
  const bool fused = !tc && gemv_fuses_combine(n_tokens);
  CombineArgs cb{};
  if (fused) {
    cb.gates = h->plan.gates;
    cb.inv = h->plan.inv;
    cb.out = reinterpret_cast<__nv_bfloat16 *>(out);
    cb.counters = h->combine_counters;
    cb.T = n_tokens;
  }
  bool down_done = false;
  // the first gate/up kernel follows the route kernel directly
  fa.pdl = !tc && !h->prof && !capturing;
  if (kcopy) {
    // misses copied on the device from the GPU's miss list (no host round
    // trip): ranges 0-1 = what the gate/up projection reads, range 2 = the rest
    const BlobLayout bl = blob_layout(h->fmt, h->H, h->I);
    MissCopyArgs &mc = fa.mc;
    mc.miss = h->plan.miss;
    mc.n = h->plan.n;
    mc.pool_dev = h->pool_dev;
    mc.slots = h->slots;
    mc.slot_stride = h->slot_stride;
    mc.seg[0][0] = 0;
    mc.seg[0][1] = bl.d_codes;
    mc.seg[1][0] = bl.gscale >= 0 ? bl.gscale : 0;
    mc.seg[1][1] = bl.gscale >= 0 ? h->blob_bytes : 0;
    mc.seg[2][0] = bl.d_codes;
    mc.seg[2][1] = bl.gscale >= 0 ? bl.gscale : h->blob_bytes;
    if (!tc) {
      // GEMV: the gate/up kernel's first grid rows copy; its miss CTAs wait
      // for their flag and the down kernel follows the whole grid
      fa.only = 0;
      const int fb = gateup_feature_blocks(h->H, h->I);
      fa.copy_rows = std::max(1, (kCopyCtas + fb - 1) / fb);
      fa.copy_sync = h->copy_sync;
      fa.seq = (int)h->seq;
      // FT_FAULT=devwait: the flag is raised with a value nobody waits for, so
      // the misses' CTAs run out their bounded wait (FT_ERR_DEVICE at the next
      // synchronising call)
      fa.seq_raised = fault("devwait") ? fa.seq ^ 0x40000000 : fa.seq;
      fa.miss_coherent = 1;   // the misses' slots fill while this grid runs
      prof_begin(h, FT_PROF_GATEUP_HIT, stream);
      FT_CUDA(h, run_ffn(h, fa, false, tc, n_tokens, stream));
      prof_end(h, FT_PROF_GATEUP_HIT, stream);
      fa.copy_rows = 0;
      fa.miss_coherent = 0;
    } else {
      // tensor cores: copy kernels on the copy stream; the misses' gate/up
      // waits for the first, the down kernel for the second
      FT_CUDA(h, cudaStreamWaitEvent(h->copy_stream, h->ev_route, 0));
      prof_begin(h, FT_PROF_MISS_COPY, h->copy_stream);
      FT_CUDA(h, launch_miss_copy(mc, 0, 2, h->copy_stream));
      FT_CUDA(h, cudaEventRecord(h->ev_copy, h->copy_stream));
      FT_CUDA(h, launch_miss_copy(mc, 2, 3, h->copy_stream));
      prof_end(h, FT_PROF_MISS_COPY, h->copy_stream);
      FT_CUDA(h, cudaEventRecord(h->ev_copy2, h->copy_stream));
      h->kernel_launches += 3;   // two copies, the misses' gate/up
      fa.only = 1;
      prof_begin(h, FT_PROF_GATEUP_HIT, stream);
      FT_CUDA(h, run_ffn(h, fa, false, tc, n_tokens, stream));
      prof_end(h, FT_PROF_GATEUP_HIT, stream);
      FT_CUDA(h, cudaStreamWaitEvent(stream, h->ev_copy, 0));
      fa.only = 2;
      prof_begin(h, FT_PROF_GATEUP_MISS, stream);
      FT_CUDA(h, run_ffn(h, fa, false, tc, n_tokens, stream));
      prof_end(h, FT_PROF_GATEUP_MISS, stream);
      FT_CUDA(h, cudaStreamWaitEvent(stream, h->ev_copy2, 0));
      copies_before_down = true;
    }
    fa.pdl = 0;
  } else if (h->mode == MODE_LRU && !pull) {
    fa.only = 1;
    prof_begin(h, FT_PROF_GATEUP_HIT, stream);
    FT_CUDA(h, run_ffn(h, fa, false, tc, n_tokens, stream));
    prof_end(h, FT_PROF_GATEUP_HIT, stream);
    fa.pdl = 0;
    if (int rc = wait_plan(h)) return rc;
    const int n_miss = h->mirror_host[1];
    // GEMV calls copy each miss in two parts, the gate/up rows first: the
    // misses' gate/up kernel starts once those have landed and runs while the
    // down rows are still crossing PCIe (it reads the NVFP4 global scales,
    // which sit in the down part, from the host blob)
    const bool two_part = !tc && n_miss <= kMissScaleArgs;
    const BlobLayout bl = blob_layout(h->fmt, h->H, h->I);
    const int64_t split = two_part ? bl.d_codes : h->blob_bytes;
    if (n_miss > 0 && !tc) {
      // the hits' down projection runs now, beside the copies; the misses'
      // follows their down bytes.  Both launches arrive on the combine counters.
      fa.only = 1;
      fa.pdl = !h->prof && !capturing;
      cb.launches = 2;
      h->kernel_launches += 1;
      prof_begin(h, FT_PROF_DOWN, stream);
      FT_CUDA(h, run_ffn(h, fa, true, tc, n_tokens, stream, cb));
      prof_end(h, FT_PROF_DOWN, stream);
      fa.pdl = 0;
    }
    if (n_miss > 0) {
      // both copy streams start after the route kernel (every earlier reader
      // of an evicted slot has finished by then); misses alternate between them
      FT_CUDA(h, cudaStreamWaitEvent(h->copy_stream, h->ev_route, 0));
      if (n_miss > 1) FT_CUDA(h, cudaStreamWaitEvent(h->copy_stream2, h->ev_route, 0));
      for (int i = 0; i < n_miss; ++i) {
        const int key = h->mirror_host[2 + i], slot = h->mirror_host[2 + h->umax + i];
        if (key < 0 || key >= h->L * h->E || slot < 0 || slot >= h->S)
          return fail(h, FT_ERR_DEVICE, "miss list entry out of range");
      }
      // part 0: [0, split) of every miss; part 1: the rest
      for (int part = 0; part < (two_part ? 2 : 1); ++part) {
        const int64_t b0 = part == 0 ? 0 : split, nb = part == 0 ? split : h->blob_bytes - split;
        if (part == 0) prof_begin(h, FT_PROF_MISS_COPY, h->copy_stream);
        for (int i = 0; i < n_miss; ++i) {
          const int key = h->mirror_host[2 + i], slot = h->mirror_host[2 + h->umax + i];
          FT_CUDA(h, cudaMemcpyAsync(h->slots + (size_t)slot * h->slot_stride + b0,
                                     static_cast<const uint8_t *>(h->pool[key]) + b0, nb, cudaMemcpyHostToDevice,
                                     (i & 1) ? h->copy_stream2 : h->copy_stream));
        }
        if (n_miss > 1) {
          FT_CUDA(h, cudaEventRecord(h->ev_copy2, h->copy_stream2));
          FT_CUDA(h, cudaStreamWaitEvent(h->copy_stream, h->ev_copy2, 0));
        }
        if (part == (two_part ? 1 : 0)) prof_end(h, FT_PROF_MISS_COPY, h->copy_stream);
        FT_CUDA(h, cudaEventRecord(h->ev_copy, h->copy_stream));
        FT_CUDA(h, cudaStreamWaitEvent(stream, h->ev_copy, 0));
        if (part == 0) {
          fa.only = 2;
          if (two_part && h->fmt == FMT_NVFP4) {
            fa.ms.n = n_miss;
            for (int i = 0; i < n_miss; ++i) {
              const int key = h->mirror_host[2 + i];
              const float *g = reinterpret_cast<const float *>(static_cast<const uint8_t *>(h->pool[key]) + bl.gscale);
              fa.ms.expert[i] = key % h->E;
              fa.ms.gate[i] = g[0];
              fa.ms.up[i] = g[1];
            }
          }
          h->kernel_launches += 1;
          prof_begin(h, FT_PROF_GATEUP_MISS, stream);
          FT_CUDA(h, run_ffn(h, fa, false, tc, n_tokens, stream));
          prof_end(h, FT_PROF_GATEUP_MISS, stream);
          fa.ms.n = 0;
        }
      }
      copies_before_down = two_part;
      if (!tc) {
        // the misses' down projection, after the last copies (no kernel between)
        fa.only = 2;
        fa.pdl = 0;
        prof_begin(h, FT_PROF_DOWN, stream);
        FT_CUDA(h, run_ffn(h, fa, true, tc, n_tokens, stream, cb));
        prof_end(h, FT_PROF_DOWN, stream);
        down_done = true;
      }
    }
  } else {
    fa.only = 0;
    prof_begin(h, FT_PROF_GATEUP_HIT, stream);
    FT_CUDA(h, run_ffn(h, fa, false, tc, n_tokens, stream));
    prof_end(h, FT_PROF_GATEUP_HIT, stream);
  }
  fa.only = 0;
  // the down kernel follows the gate/up kernel directly (unless it waits for copies)
  fa.pdl = !tc && !h->prof && !capturing && !copies_before_down;
  if (tc) {
    // tensor cores: the down GEMM adds each row, gate-weighted, into the
    // fp32 output rows; y reaches memory only when activations are kept
    fa.out_acc = h->out_acc;
    fa.keep_y = h->keep_y ? 1 : 0;
    FT_CUDA(h, cudaMemsetAsync(h->out_acc, 0, sizeof(float) * (size_t)n_tokens * h->H, stream));
  }
  if (!down_done) {
    prof_begin(h, FT_PROF_DOWN, stream);
    FT_CUDA(h, run_ffn(h, fa, true, tc, n_tokens, stream, cb));
    prof_end(h, FT_PROF_DOWN, stream);
  }
  if (tc) {
    h->kernel_launches += 1;
    prof_begin(h, FT_PROF_COMBINE, stream);
    FT_CUDA(h, launch_acc_to_bf16(h->out_acc, reinterpret_cast<__nv_bfloat16 *>(out), (int64_t)n_tokens * h->H,
                                  stream));
    prof_end(h, FT_PROF_COMBINE, stream);
  } else if (!fused) {
    h->kernel_launches += 1;
    prof_begin(h, FT_PROF_COMBINE, stream);
    FT_CUDA(h, launch_combine(h->ybuf, h->plan.gates, h->plan.inv, n_tokens, h->k, h->H,
                              reinterpret_cast<__nv_bfloat16 *>(out), stream));
    prof_end(h, FT_PROF_COMBINE, stream);
  }
  if (h->mode == MODE_STREAM) FT_CUDA(h, cudaEventRecord(h->ev_bank_free[bank], stream));
  // a captured call runs when its graph is launched: the next synchronising
  // call waits for the device instead of the handle's event
  if (capturing) h->captured = true;
  else FT_CUDA(h, cudaEventRecord(h->ev_done, stream));
  h->host_streamed += h->last_streamed;
  h->host_bytes += h->last_stream_bytes;
  h->host_d2d += h->last_d2d;
  return FT_OK;
}

int ft_moe_set_profiling(ft_moe *h, int enable) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (int rc = sync_handle(h)) return rc;
  if (enable)
    for (auto &cls : h->prof_ev)
      for (auto &pair : cls)
        for (cudaEvent_t &ev : pair)
          if (!ev) FT_CUDA(h, cudaEventCreate(&ev));
  for (int c = 0; c < FT_PROF_CLASSES; ++c) {
    h->prof_ms[c] = 0.0;
    h->prof_launches[c] = 0;
    h->prof_head[c] = 0;
    h->prof_count[c] = 0;
  }
  h->prof = enable != 0;
  return FT_OK;
}

int ft_moe_profile_read(ft_moe *h, double *ms, int64_t *launches, int n) {
  if (!h || n < 0) return fail(h, FT_ERR_ARG, "NULL handle or negative n");
  if (int rc = sync_handle(h)) return rc;
  prof_collect(h);
  for (int c = 0; c < std::min(n, (int)FT_PROF_CLASSES); ++c) {
    if (ms) ms[c] = h->prof_ms[c];
    if (launches) launches[c] = h->prof_launches[c];
  }
  return FT_OK;
}

int ft_cache_stats(ft_moe *h, ft_stats *cum, ft_stats *last) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (int rc = sync_handle(h)) return rc;
  unsigned long long d[16];
  FT_CUDA(h, cudaMemcpy(d, h->stats_dev, sizeof d, cudaMemcpyDeviceToHost));
  if (cum) *cum = ft_stats{d[0], d[1], d[2], d[3], h->host_warm, h->host_streamed, d[4] + h->host_bytes, h->host_d2d};
  if (last) {
    if (h->last_T == 0) *last = ft_stats{0, 0, 0, 0, 0, 0, 0, 0};
    else *last = ft_stats{d[8], d[9], d[10], d[11], 0, h->last_streamed, d[12] + h->last_stream_bytes, h->last_d2d};
  }
  return FT_OK;
}

int ft_cache_trace(ft_moe *h, int32_t *experts, int32_t *slots, int32_t *hit, int32_t *evicted, int cap, int *n) {
  if (!h || cap < 0) return fail(h, FT_ERR_ARG, "NULL handle or negative cap");
  if (int rc = sync_handle(h)) return rc;
  int cnt[4] = {0, 0, 0, 0};
  if (h->last_T > 0) FT_CUDA(h, cudaMemcpy(cnt, h->plan.n, sizeof cnt, cudaMemcpyDeviceToHost));
  const int m = std::min(cap, cnt[0]);
  if (m > 0) {
    if (experts) FT_CUDA(h, cudaMemcpy(experts, h->plan.u_expert, 4 * (size_t)m, cudaMemcpyDeviceToHost));
    if (slots) FT_CUDA(h, cudaMemcpy(slots, h->plan.u_slot, 4 * (size_t)m, cudaMemcpyDeviceToHost));
    if (hit) FT_CUDA(h, cudaMemcpy(hit, h->plan.u_hit, 4 * (size_t)m, cudaMemcpyDeviceToHost));
    if (evicted) FT_CUDA(h, cudaMemcpy(evicted, h->plan.u_evicted, 4 * (size_t)m, cudaMemcpyDeviceToHost));
  }
  if (n) *n = cnt[0];
  return FT_OK;
}

int ft_moe_last_routing(ft_moe *h, int32_t *topk_idx, float *gates, int32_t *offsets, int32_t *perm, int32_t *inv,
                        int *n_tokens) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (int rc = sync_handle(h)) return rc;
  const size_t TK = (size_t)h->last_T * h->k;
  if (TK) {
    if (topk_idx) FT_CUDA(h, cudaMemcpy(topk_idx, h->plan.topk_idx, 4 * TK, cudaMemcpyDeviceToHost));
    if (gates) FT_CUDA(h, cudaMemcpy(gates, h->plan.gates, 4 * TK, cudaMemcpyDeviceToHost));
    if (offsets) FT_CUDA(h, cudaMemcpy(offsets, h->plan.offsets, 4 * (size_t)(h->E + 1), cudaMemcpyDeviceToHost));
    if (perm) FT_CUDA(h, cudaMemcpy(perm, h->plan.perm, 4 * TK, cudaMemcpyDeviceToHost));
    if (inv) FT_CUDA(h, cudaMemcpy(inv, h->plan.inv, 4 * TK, cudaMemcpyDeviceToHost));
  }
  if (n_tokens) *n_tokens = h->last_T;
  return FT_OK;
}

int ft_moe_last_activations(ft_moe *h, uint16_t *h_act, float *y) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (int rc = sync_handle(h)) return rc;
  const size_t TK = (size_t)h->last_T * h->k;
  if (TK && h_act) FT_CUDA(h, cudaMemcpy(h_act, h->hbuf, 2 * TK * h->I, cudaMemcpyDeviceToHost));
  if (TK && y) FT_CUDA(h, cudaMemcpy(y, h->ybuf, 4 * TK * h->H, cudaMemcpyDeviceToHost));
  return FT_OK;
}

int ft_moe_set_ffn_kernel(ft_moe *h, int which) {
  if (!h || which < FT_FFN_AUTO || which > FT_FFN_TC) return fail(h, FT_ERR_ARG, "bad FFN kernel choice");
  if (which == FT_FFN_TC && !h->tmaps_ok)
    return fail(h, FT_ERR_CUDA, "tensor-core FFN unavailable: the TMA descriptors could not be encoded");
  h->ffn_kernel = which;
  return FT_OK;
}

int ft_moe_last_ffn_kernel(const ft_moe *h) { return h ? (h->last_tc ? FT_FFN_TC : FT_FFN_GEMV) : -1; }

int ft_moe_miss_path(const ft_moe *h, int tensor_core) { return h ? effective_miss_path(h, tensor_core != 0) : -1; }

int ft_moe_set_keep_activations(ft_moe *h, int on) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (int rc = sync_handle(h)) return rc;
  h->keep_y = on != 0;
  return FT_OK;
}

int ft_moe_set_decode_fusion(ft_moe *h, int on) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (int rc = sync_handle(h)) return rc;
  h->decode_fused = on != 0;
  return FT_OK;
}

int ft_moe_set_decode_grid(ft_moe *h, int on) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (int rc = sync_handle(h)) return rc;
  h->decode_grid = on != 0;
  return FT_OK;
}

int ft_moe_set_miss_path(ft_moe *h, int path) {
  if (!h || path < FT_MISS_COPY || path > FT_MISS_AUTO)
    return fail(h, FT_ERR_ARG, "bad miss path");
  if (int rc = sync_handle(h)) return rc;
  h->miss_path = path;
  return FT_OK;
}

// FP4 x FP4 variant ("The Real Requirement Is System RAM": NVFP4 = 4-bit
// values with an 8-bit scale per 16 weights; the activations take the same
// layout here).  Buffers over expert-padded rows are allocated on first use.
int ft_moe_set_act_format(ft_moe *h, int act_fmt) {
  if (!h || (act_fmt != FT_ACT_BF16 && act_fmt != FT_ACT_FP4)) return fail(h, FT_ERR_ARG, "NULL handle or bad act_fmt");
  if (int rc = sync_handle(h)) return rc;
  if (act_fmt == FT_ACT_BF16) {
    h->act_fmt = act_fmt;
    return FT_OK;
  }
  if (h->fmt != FMT_NVFP4) return fail(h, FT_ERR_ARG, "FP4 activations need NVFP4 weights");
  FT_CUDA(h, cudaSetDevice(h->device));
  if (!h->q.xq) {
    const int64_t rows = fp4_padded_rows((int64_t)h->Tmax * h->k, h->umax);
    Fp4Bufs q{};
    const bool ok = cudaMalloc(&q.xq, (size_t)rows * h->H / 2) == cudaSuccess &&
                    cudaMalloc(&q.xsf, (size_t)rows * h->H / 16) == cudaSuccess &&
                    cudaMalloc(&q.xg, (size_t)rows * sizeof(float)) == cudaSuccess &&
                    cudaMalloc(&q.hq, (size_t)rows * h->I / 2) == cudaSuccess &&
                    cudaMalloc(&q.hsf, (size_t)rows * h->I / 16) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      cudaFree(q.xq);
      cudaFree(q.xsf);
      cudaFree(q.xg);
      cudaFree(q.hq);
      cudaFree(q.hsf);
      return fail(h, FT_ERR_OOM, "device allocation of the FP4 activation buffers failed");
    }
    h->q = q;
    h->q_rows = rows;
    h->qmaps_ok = make_fp4_maps(h->slots, h->slot_stride, h->S, h->H, h->I, h->q.xq, h->q.hq, rows, h->qmap[0],
                                h->qmap[1], h->qmap[2], h->qmap[3], h->qmap[4], h->qmap[5]) == 0;
  }
  if (!h->qmaps_ok) return fail(h, FT_ERR_CUDA, "FP4 TMA descriptors could not be encoded");
  h->act_fmt = act_fmt;
  return FT_OK;
}

int ft_moe_act_format(const ft_moe *h) { return h ? h->act_fmt : -1; }

int ft_moe_last_act_fp4(ft_moe *h, uint8_t *x_codes, uint8_t *x_sf, float *x_g, uint8_t *h_codes, uint8_t *h_sf) {
  if (!h) return fail(h, FT_ERR_ARG, "NULL handle");
  if (int rc = sync_handle(h)) return rc;
  if (!h->q.xq || !h->last_tc || h->act_fmt != FT_ACT_FP4)
    return fail(h, FT_ERR_STATE, "the last forward did not run the FP4 x FP4 FFN");
  const int T = h->last_T, k = h->k, E = h->E, H = h->H, I = h->I;
  const size_t TK = (size_t)T * k;
  if (TK == 0) return FT_OK;
  std::vector<int32_t> off(E + 1);
  FT_CUDA(h, cudaMemcpy(off.data(), h->plan.offsets, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToHost));
  std::vector<int64_t> pad(E + 1, 0);
  for (int e = 0; e < E; ++e) pad[e + 1] = pad[e] + (off[e + 1] - off[e] + 127) / 128 * 128;
  const int64_t rows = pad[E];
  std::vector<uint8_t> xq((size_t)rows * H / 2), xsf((size_t)rows * H / 16), hq((size_t)rows * I / 2),
      hsf((size_t)rows * I / 16);
  std::vector<float> xg(rows);
  FT_CUDA(h, cudaMemcpy(xq.data(), h->q.xq, xq.size(), cudaMemcpyDeviceToHost));
  FT_CUDA(h, cudaMemcpy(xsf.data(), h->q.xsf, xsf.size(), cudaMemcpyDeviceToHost));
  FT_CUDA(h, cudaMemcpy(xg.data(), h->q.xg, xg.size() * sizeof(float), cudaMemcpyDeviceToHost));
  FT_CUDA(h, cudaMemcpy(hq.data(), h->q.hq, hq.size(), cudaMemcpyDeviceToHost));
  FT_CUDA(h, cudaMemcpy(hsf.data(), h->q.hsf, hsf.size(), cudaMemcpyDeviceToHost));
  auto atom = [](int64_t r, int b, int K) {
    return ((size_t)(r >> 7) * (K >> 6) + (b >> 2)) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3) + (b & 3);
  };
  for (int e = 0; e < E; ++e)
    for (int p = off[e]; p < off[e + 1]; ++p) {
      const int64_t r = pad[e] + (p - off[e]);
      if (x_codes) std::memcpy(x_codes + (size_t)p * H / 2, xq.data() + (size_t)r * H / 2, H / 2);
      if (h_codes) std::memcpy(h_codes + (size_t)p * I / 2, hq.data() + (size_t)r * I / 2, I / 2);
      if (x_g) x_g[p] = xg[r];
      if (x_sf)
        for (int b = 0; b < H / 16; ++b) x_sf[(size_t)p * (H / 16) + b] = xsf[atom(r, b, H)];
      if (h_sf)
        for (int b = 0; b < I / 16; ++b) h_sf[(size_t)p * (I / 16) + b] = hsf[atom(r, b, I)];
    }
  return FT_OK;
}

int64_t ft_moe_slot_stride(const ft_moe *h) { return h ? h->slot_stride : -1; }

int64_t ft_moe_kernel_launches(const ft_moe *h) { return h ? h->kernel_launches : -1; }

const char *ft_last_error(const ft_moe *h) { return h ? h->err.c_str() : g_create_err.c_str(); }

int ft_moe_destroy(ft_moe *h) {
  if (!h) return FT_OK;
  cudaSetDevice(h->device);
  sync_handle(h);
  free_all(h);
  delete h;
  return FT_OK;
}

int ft_topk_softmax(const float *router_logits, int T, int E, int k, int32_t *topk_idx, float *gates, void *stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || k > std::min(E, kMaxTopK))
    return fail(nullptr, FT_ERR_ARG, "bad T/E/k");
  if (T > 0 && (!router_logits || !topk_idx || !gates)) return fail(nullptr, FT_ERR_ARG, "NULL pointer");
  cudaError_t e = launch_topk_only(router_logits, T, E, k, topk_idx, gates, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FT_OK : cuda_fail(nullptr, e, "topk kernel");
}

int ft_fp4_tensor_peak(int n_tile, int iters, double *tflops) {
  if ((n_tile != 128 && n_tile != 256) || iters < 1 || !tflops)
    return fail(nullptr, FT_ERR_ARG, "n_tile must be 128 or 256, iters >= 1, tflops not NULL");
  int *err = nullptr;
  if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return fail(nullptr, FT_ERR_OOM, "device allocation failed");
  }
  cudaMemset(err, 0, sizeof(int));
  fp4_init_attributes();
  const double ms = fp4_peak_ms(n_tile, iters, err, nullptr);
  int code = 0;
  cudaError_t e = cudaMemcpy(&code, err, sizeof code, cudaMemcpyDeviceToHost);
  cudaFree(err);
  if (ms < 0 || e != cudaSuccess) return cuda_fail(nullptr, e != cudaSuccess ? e : cudaGetLastError(), "fp4 peak kernel");
  if (code != 0) return fail(nullptr, FT_ERR_DEVICE, "fp4 peak kernel gave up its bounded wait");
  const double flops = (double)tc_num_sms() * iters * 4 * 2.0 * 128 * n_tile * 64;
  *tflops = flops / (ms * 1e-3) / 1e12;
  return FT_OK;
}

size_t ft_permute_workspace_bytes(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  return sizeof(int32_t) * permute_scratch_ints(T, k, E);
}

int ft_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *offsets, int32_t *perm, int32_t *inv,
               void *workspace, size_t workspace_bytes, void *stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || k > kMaxTopK) return fail(nullptr, FT_ERR_ARG, "bad T/E/k");
  if (!offsets || (T > 0 && (!topk_idx || !perm || !inv))) return fail(nullptr, FT_ERR_ARG, "NULL pointer");
  const size_t need = ft_permute_workspace_bytes(T, k, E);
  if (need > 0 && (!workspace || workspace_bytes < need)) return fail(nullptr, FT_ERR_ARG, "workspace too small");
  int32_t *ws = reinterpret_cast<int32_t *>(workspace);
  const size_t half = permute_scratch_ints(T, k, E) / 2;
  cudaError_t e = launch_permute_only(topk_idx, T, k, E, offsets, perm, inv, ws, ws ? ws + half : nullptr,
                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FT_OK : cuda_fail(nullptr, e, "permute kernels");
}

}  // extern "C"
