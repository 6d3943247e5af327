// route_dev.cuh -- device code of the routing step (top-k + softmax, permute,
// on-device LRU plan), shared by the routing kernels and the fused decode
// layer kernel.  See route.cu for the design.
#pragma once
#include <math.h>

#include "ft_internal.cuh"

namespace ftmoe {
namespace {


__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive block-wide prefix sum of v; *total receives the block sum.
// All threads of the block must call it.  s_warp holds >= 32 ints.
__device__ int block_excl_scan(int v, int *s_warp, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    s_warp[lane] = t;
  }
  __syncthreads();
  const int base = w ? s_warp[w - 1] : 0;
  *total = s_warp[nw - 1];
  __syncthreads();
  return base + x - v;
}

// Order-preserving map of a float to an unsigned key (larger float, larger
// key); +0 and -0 map to the same key.  key_of(-inf) = 0x007FFFFF > 0, so a
// key of 0 marks "taken or padding".
__device__ __forceinline__ uint32_t key_of(float x) {
  if (x == 0.0f) x = 0.0f;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float float_of(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp selects the k largest logits of one token (ties to the lower id,
// NaN treated as -inf) and writes their ids and softmax gates.  Lane l holds
// experts l, l+32, ..; each round takes the warp-wide largest key (redux.sync)
// and, among lanes holding it, the lowest expert id (a second redux).
// Returns, in lanes 0..k-1, the selected expert of rank `lane` (else -1).
template <int NV>
__device__ int warp_topk_softmax_t(const float *__restrict__ row, int E, int k, int32_t *out_idx, float *out_gate) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    float x = e < E ? __ldg(row + e) : -INFINITY;
    if (isnan(x)) x = -INFINITY;
    key[i] = e < E ? key_of(x) : 0u;
  }
  auto local_best = [&](uint32_t &bk, int &bi) {
    bk = 0u;
    bi = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (key[i] > bk) {   // strict: the lowest i (lowest id) keeps a tie
        bk = key[i];
        bi = i;
      }
  };
  uint32_t bk;
  int bi;
  local_best(bk, bi);
  float my_v = -INFINITY;
  int my_i = -1;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t cand = bk == m ? (uint32_t)(lane + 32 * bi) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if (lane == (int)(win & 31u)) {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (i == (int)(win >> 5)) key[i] = 0u;
      local_best(bk, bi);
    }
    if (lane == j) {
      my_v = float_of(m);
      my_i = (int)win;
    }
  }
  const float mx = __shfl_sync(0xffffffffu, my_v, 0);
  float z = lane < k ? expf(my_v - mx) : 0.0f;
  float sum = z;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    out_idx[lane] = my_i;
    out_gate[lane] = z / sum;
  }
  return lane < k ? my_i : -1;
}

__device__ __forceinline__ int warp_topk_softmax(const float *__restrict__ row, int E, int k, int32_t *out_idx,
                                                 float *out_gate) {
  if (E <= 32) return warp_topk_softmax_t<1>(row, E, k, out_idx, out_gate);
  if (E <= 64) return warp_topk_softmax_t<2>(row, E, k, out_idx, out_gate);
  if (E <= 128) return warp_topk_softmax_t<4>(row, E, k, out_idx, out_gate);
  if (E <= 256) return warp_topk_softmax_t<8>(row, E, k, out_idx, out_gate);
  return warp_topk_softmax_t<kMaxExperts / 32>(row, E, k, out_idx, out_gate);
}

// Stable scatter of pairs [p0, p1) by expert.  s_base[e] is the next free
// permuted position of expert e and is advanced.  s_wcnt holds nwarps*E ints.
__device__ void block_rank_scatter(const int32_t *__restrict__ idx, int p0, int p1, int E, int *s_base,
                                   int *s_wcnt, int32_t *__restrict__ perm, int32_t *__restrict__ inv) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
  if (p1 - p0 <= 32) {
    // one warp: rank among equal ids by lane order
    if (w == 0) {
      const int p = p0 + lane;
      int e = p < p1 ? idx[p] : -1;
      const bool valid = e >= 0 && e < E;
      if (!valid) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (valid) {
        const int pos = s_base[e] + __popc(peers & lanemask_lt());
        perm[pos] = p;
        inv[p] = pos;
      }
      __syncwarp();
      if (valid && lane == __ffs(peers) - 1) s_base[e] += __popc(peers);
    }
    __syncthreads();
    return;
  }
  for (int r0 = p0; r0 < p1; r0 += blockDim.x) {
    for (int i = tid; i < nw * E; i += blockDim.x) s_wcnt[i] = 0;
    __syncthreads();
    const int p = r0 + tid;
    int e = p < p1 ? idx[p] : -1;
    const bool valid = e >= 0 && e < E;   // out-of-range ids are not placed
    if (!valid) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & lanemask_lt());
    if (valid && lane == __ffs(peers) - 1) s_wcnt[w * E + e] = __popc(peers);
    __syncthreads();
    for (int e2 = tid; e2 < E; e2 += blockDim.x) {
      int run = s_base[e2];
      for (int ww = 0; ww < nw; ++ww) {
        const int c = s_wcnt[ww * E + e2];
        s_wcnt[ww * E + e2] = run;
        run += c;
      }
      s_base[e2] = run;
    }
    __syncthreads();
    if (valid) {
      const int pos = s_wcnt[w * E + e] + rank_w;
      perm[pos] = p;
      inv[p] = pos;
    }
    __syncthreads();
  }
}

struct PlanSmem {
  int *s_count;   // [E] tokens per expert in this call
  int *s_uexp;    // [E]
  int *s_victim;  // [E]
  unsigned *s_bits;  // [(S+31)/32]
  int *s_warp;    // [33]: scan partials, [32] a counter
  int *s_keyslot;    // [E] this layer's key -> slot, loaded up front (or null)
  int *s_victim_key; // [E] key held by each victim slot (with s_keyslot)
  const int *s_off;  // [E] first permuted position of each expert
};

// The cache-table entries a thread needs, loaded at kernel start so that the
// plan itself waits on no global memory: its range of the recency list and the
// key held by each of those slots.
constexpr int kPre = 8;
struct Prefetch {
  int n;              // entries held, or -1 (range longer than kPre: read in place)
  int ord[kPre], key[kPre];
  unsigned long long st[5];   // thread 0: the cumulative counters
};

__device__ __forceinline__ void prefetch_tables(const RouteArgs &a, int *s_keyslot, Prefetch &pf) {
  const int tid = threadIdx.x, NT = blockDim.x;
  pf.n = -1;
  if (tid == 0)
    for (int i = 0; i < 5; ++i) pf.st[i] = a.cache.stats[i];
  if (a.mode != MODE_LRU) return;
  for (int e = tid; e < a.E; e += NT) s_keyslot[e] = a.cache.key_slot[a.layer * a.E + e];
  const int per = (a.S + NT - 1) / NT;
  if (per > kPre) return;
  const int i0 = min(a.S, tid * per), i1 = min(a.S, i0 + per);
  pf.n = i1 - i0;
#pragma unroll
  for (int q = 0; q < kPre; ++q)
    if (q < pf.n) pf.ord[q] = a.cache.order_in[i0 + q];
#pragma unroll
  for (int q = 0; q < kPre; ++q)
    if (q < pf.n) pf.key[q] = a.cache.slot_key[pf.ord[q]];
}

// Distinct experts of the call, slot lookup, LRU update, plan and stats.
// One CTA.  Needs blockDim.x >= E.  With a prefetch (pf.n >= 0 and
// sm.s_keyslot set), the tables are read from what prefetch_tables loaded.
// The miss list is published to the host before the statistics are updated.
__device__ void block_plan(const RouteArgs &a, const PlanSmem &sm, const Prefetch &pf) {
  const int tid = threadIdx.x, NT = blockDim.x, E = a.E, S = a.S;
  const int flag = (tid < E) && sm.s_count[tid] > 0;
  int nU;
  const int u = block_excl_scan(flag, sm.s_warp, &nU);
  if (flag) sm.s_uexp[u] = tid;
  __syncthreads();

  int key = -1, slot = -1, hit = 0;
  if (tid < nU) {
    const int e = sm.s_uexp[tid];
    key = a.layer * E + e;
    if (a.mode == MODE_LRU) {
      slot = sm.s_keyslot ? sm.s_keyslot[e] : a.cache.key_slot[key];
      hit = slot >= 0;
    } else {
      slot = a.bank_slot0 + e;
      hit = 1;
    }
  }
  int nH;
  const int hrank = block_excl_scan(tid < nU && hit, sm.s_warp, &nH);
  const int nM = nU - nH;
  const int mrank = tid - hrank;
  int evicted = -1;

  if (a.mode == MODE_LRU) {
    const int nwords = (S + 31) >> 5;
    for (int i = tid; i < nwords; i += NT) sm.s_bits[i] = 0u;
    __syncthreads();
    if (tid < nU && hit) atomicOr(&sm.s_bits[slot >> 5], 1u << (slot & 31));
    __syncthreads();
    const int per = (S + NT - 1) / NT;
    const int i0 = min(S, tid * per), i1 = min(S, i0 + per);
    int cnt = 0, r;
    if (pf.n >= 0) {
#pragma unroll
      for (int q = 0; q < kPre; ++q)
        if (q < pf.n) cnt += !((sm.s_bits[pf.ord[q] >> 5] >> (pf.ord[q] & 31)) & 1u);
      int nonhit;
      r = block_excl_scan(cnt, sm.s_warp, &nonhit);
#pragma unroll
      for (int q = 0; q < kPre; ++q) {
        if (q >= pf.n) continue;
        const int s = pf.ord[q];
        if ((sm.s_bits[s >> 5] >> (s & 31)) & 1u) continue;
        if (r < nM) {
          sm.s_victim[r] = s;
          sm.s_victim_key[r] = pf.key[q];
        } else {
          a.cache.order_out[r - nM] = s;
        }
        ++r;
      }
    } else {
      for (int i = i0; i < i1; ++i) {
        const int s = a.cache.order_in[i];
        cnt += !((sm.s_bits[s >> 5] >> (s & 31)) & 1u);
      }
      int nonhit;
      r = block_excl_scan(cnt, sm.s_warp, &nonhit);
      for (int i = i0; i < i1; ++i) {
        const int s = a.cache.order_in[i];
        if ((sm.s_bits[s >> 5] >> (s & 31)) & 1u) continue;
        if (r < nM) sm.s_victim[r] = s;
        else a.cache.order_out[r - nM] = s;
        ++r;
      }
    }
    __syncthreads();
    if (tid < nU) {
      if (hit) {
        a.cache.order_out[S - nH - nM + hrank] = slot;
      } else {
        const int v = sm.s_victim[mrank];
        a.cache.order_out[S - nM + mrank] = v;
        const int ek = pf.n >= 0 ? sm.s_victim_key[mrank] : a.cache.slot_key[v];
        if (ek >= 0) {
          a.cache.key_slot[ek] = -1;
          evicted = ek;
        }
        a.cache.slot_key[v] = key;
        a.cache.key_slot[key] = v;
        slot = v;
      }
    }
  }
  // evictions of this call: a count in shared memory (no order needed)
  if (tid == 0) sm.s_warp[32] = 0;
  __syncthreads();
  if (evicted >= 0) atomicAdd(&sm.s_warp[32], 1);
  __syncthreads();
  const int nEv = sm.s_warp[32];
  if (tid < nU) {
    a.plan.u_expert[tid] = sm.s_uexp[tid];
    a.plan.u_slot[tid] = slot;
    a.plan.u_hit[tid] = hit;
    a.plan.u_evicted[tid] = evicted;
    // hits first: the GEMV grid's rows follow this order, so that CTAs that
    // wait for a miss's bytes are dispatched after every hit's CTAs
    const int e = sm.s_uexp[tid];
    a.plan.u_info[hit ? hrank : nH + mrank] = make_int4(e, slot, sm.s_off[e], (sm.s_count[e] << 1) | hit);
    if (!hit) {
      a.plan.miss[mrank] = make_int2(key, slot);
      if (a.mirror) {
        a.mirror[2 + mrank] = key;
        a.mirror[2 + a.umax + mrank] = slot;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (a.mirror) {
      // the block's miss-list writes precede this fence (barrier above), and
      // the host reads the list only after it sees the new sequence number
      a.mirror[1] = nM;
      __threadfence_system();
      *(volatile int32_t *)&a.mirror[0] = (int32_t)a.seq;
    }
    a.plan.n[0] = nU;
    a.plan.n[1] = nH;
    a.plan.n[2] = nM;
    a.plan.n[3] = nEv;
    unsigned long long *st = a.cache.stats;
    const unsigned long long bytes = a.mode == MODE_LRU ? (unsigned long long)nM * a.blob_bytes : 0ull;
    const unsigned long long hits_ = a.mode == MODE_LRU ? nH : 0, miss_ = a.mode == MODE_LRU ? nM : 0;
    st[0] = pf.st[0] + nU; st[1] = pf.st[1] + hits_; st[2] = pf.st[2] + miss_; st[3] = pf.st[3] + nEv;
    st[4] = pf.st[4] + bytes;
    st[8] = nU; st[9] = hits_; st[10] = miss_; st[11] = nEv; st[12] = bytes;
  }
}

// Whole routing of a small call in one CTA: top-k + gates, histogram,
// offsets, plan, stable scatter.  The cache tables are read at the start,
// alongside the logits, so the plan waits on no further global loads.
__device__ __forceinline__ void route_small_body(const RouteArgs &a, int *smem, bool pdl) {
  const int E = a.E, nw = blockDim.x >> 5;
  int *s_count = smem;                 // E
  int *s_base = s_count + E;           // E
  int *s_uexp = s_base + E;            // E
  int *s_victim = s_uexp + E;          // E
  int *s_keyslot = s_victim + E;       // E
  int *s_victim_key = s_keyslot + E;   // E
  int *s_warp = s_victim_key + E;      // 33
  int *s_wcnt = s_warp + 33;           // nw*E
  unsigned *s_bits = (unsigned *)(s_wcnt + nw * E);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  // the cache tables were last written by the previous call's route kernel,
  // which has completed (see pdl_trigger); everything else waits for the
  // kernel before this one
  Prefetch pf;
  prefetch_tables(a, s_keyslot, pf);
  if (pdl) {
    pdl_wait();
    pdl_trigger();
  }
  for (int i = tid; i < E; i += blockDim.x) s_count[i] = 0;
  __syncthreads();
  for (int t = w; t < a.T; t += nw) {
    const int e = warp_topk_softmax(a.logits + (size_t)t * E, E, a.k, a.plan.topk_idx + (size_t)t * a.k,
                                    a.plan.gates + (size_t)t * a.k);
    if (lane < a.k) atomicAdd(&s_count[e], 1);
  }
  __syncthreads();
  int total;
  const int off = block_excl_scan(tid < E ? s_count[tid] : 0, s_warp, &total);
  if (tid < E) {
    a.plan.offsets[tid] = off;
    s_base[tid] = off;
  }
  if (tid == 0) a.plan.offsets[E] = total;
  PlanSmem sm{s_count, s_uexp, s_victim, s_bits, s_warp, a.mode == MODE_LRU ? s_keyslot : nullptr, s_victim_key,
              s_base};
  block_plan(a, sm, pf);
  __syncthreads();
  block_rank_scatter(a.plan.topk_idx, 0, a.T * a.k, E, s_base, s_wcnt, a.plan.perm, a.plan.inv);
}


// Routing of a decode-sized call (T*k <= 32 pairs) in one CTA with four
// block barriers instead of the general path's two dozen: the warps take one
// token each for the top-k; warp 0 alone derives the offsets, the distinct
// experts, the hits and the stable permute (one pair per lane); all threads
// compact the recency list; warp 0 finishes the plan.  Same results, in the
// same order, as route_small_body.
constexpr int kDecodeRoutePairs = 32;
__device__ __forceinline__ void route_decode_body(const RouteArgs &a, int *smem, bool pdl) {
  const int E = a.E, S = a.S, P = a.T * a.k;
  const int nw = blockDim.x >> 5;
  const bool lru = a.mode == MODE_LRU;
  int *s_count = smem;                 // E   tokens per expert
  int *s_off = s_count + E;            // E   first permuted position per expert
  int *s_uexp = s_off + E;             // E   distinct experts, ascending
  int *s_victim = s_uexp + E;          // E
  int *s_keyslot = s_victim + E;       // E
  int *s_victim_key = s_keyslot + E;   // E
  int *s_wt = s_victim_key + E;        // 33  per-warp totals
  int *s_pe = s_wt + 33;               // 32  expert of each pair
  int *s_uslot = s_pe + 32;            // 32  slot of each distinct expert (-1: miss)
  int *s_sc = s_uslot + 32;            // 4   nU, nH, nM
  unsigned *s_bits = (unsigned *)(s_sc + 4);   // [S/32] hit slots
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  Prefetch pf;
  prefetch_tables(a, s_keyslot, pf);
  // the call's logits (an input, final before the kernel ahead, which writes
  // only the previous call's output) are asked into L2 before the wait
  for (int i = tid * 32; i < a.T * E; i += blockDim.x * 32)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.logits + i));
  if (pdl) {
    pdl_wait();
    pdl_trigger();
  }
  for (int i = tid; i < E; i += blockDim.x) s_count[i] = 0;
  if (lru)
    for (int i = tid; i < ((S + 31) >> 5); i += blockDim.x) s_bits[i] = 0u;
  __syncthreads();
  for (int t = w; t < a.T; t += nw) {
    const int e = warp_topk_softmax(a.logits + (size_t)t * E, E, a.k, a.plan.topk_idx + (size_t)t * a.k,
                                    a.plan.gates + (size_t)t * a.k);
    if (lane < a.k) {
      atomicAdd(&s_count[e], 1);
      s_pe[t * a.k + lane] = e;
    }
  }
  __syncthreads();
  if (w == 0) {
    // offsets and distinct experts: lane l scans experts [l*per, (l+1)*per)
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int c = 0, d = 0;
    for (int e = e0; e < e1; ++e) {
      const int n = s_count[e];
      c += n;
      d += n > 0;
    }
    int ci = c, di = d;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ci, o), z = __shfl_up_sync(0xffffffffu, di, o);
      if (lane >= o) {
        ci += y;
        di += z;
      }
    }
    const int total = __shfl_sync(0xffffffffu, ci, 31), nU = __shfl_sync(0xffffffffu, di, 31);
    int run = ci - c, u = di - d;
    for (int e = e0; e < e1; ++e) {
      const int n = s_count[e];
      a.plan.offsets[e] = run;
      s_off[e] = run;
      if (n > 0) s_uexp[u++] = e;
      run += n;
    }
    if (lane == 0) a.plan.offsets[E] = total;
    __syncwarp();
    // stable permute: pair p (lane p) goes to its expert's first position
    // plus the number of earlier pairs of the same expert
    const int pe = lane < P ? s_pe[lane] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, pe);
    if (lane < P) {
      const int pos = s_off[pe] + __popc(peers & lanemask_lt());
      a.plan.perm[pos] = lane;
      a.plan.inv[lane] = pos;
    }
    // hits: the distinct experts already in a slot
    int slot = -1, hit = 0;
    if (lane < nU) {
      const int eu = s_uexp[lane];
      if (lru) {
        slot = s_keyslot[eu];
        hit = slot >= 0;
      } else {
        slot = a.bank_slot0 + eu;
        hit = 1;
      }
    }
    const int nH = __popc(__ballot_sync(0xffffffffu, lane < nU && hit));
    if (lru && lane < nU && hit) atomicOr(&s_bits[slot >> 5], 1u << (slot & 31));
    s_uslot[lane] = slot;
    if (lane == 0) {
      s_sc[0] = nU;
      s_sc[1] = nH;
      s_sc[2] = nU - nH;
    }
  }
  __syncthreads();
  const int nU = s_sc[0], nH = s_sc[1], nM = s_sc[2];
  if (lru) {
    // recency list: the non-hit entries keep their order; the first nM of
    // them are the victims, the rest move to the front of the new list
    const int NT = blockDim.x;
    const int per = (S + NT - 1) / NT;
    const int i0 = min(S, tid * per), i1 = min(S, i0 + per);
    int cnt = 0;
    if (pf.n >= 0) {
#pragma unroll
      for (int q = 0; q < kPre; ++q)
        if (q < pf.n) cnt += !((s_bits[pf.ord[q] >> 5] >> (pf.ord[q] & 31)) & 1u);
    } else {
      for (int i = i0; i < i1; ++i) {
        const int sl = a.cache.order_in[i];
        cnt += !((s_bits[sl >> 5] >> (sl & 31)) & 1u);
      }
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_wt[w] = x;
    __syncthreads();
    int r = x - cnt;
    for (int ww = 0; ww < w; ++ww) r += s_wt[ww];
    if (pf.n >= 0) {
#pragma unroll
      for (int q = 0; q < kPre; ++q) {
        if (q >= pf.n) continue;
        const int sl = pf.ord[q];
        if ((s_bits[sl >> 5] >> (sl & 31)) & 1u) continue;
        if (r < nM) {
          s_victim[r] = sl;
          s_victim_key[r] = pf.key[q];
        } else {
          a.cache.order_out[r - nM] = sl;
        }
        ++r;
      }
    } else {
      for (int i = i0; i < i1; ++i) {
        const int sl = a.cache.order_in[i];
        if ((s_bits[sl >> 5] >> (sl & 31)) & 1u) continue;
        if (r < nM) {
          s_victim[r] = sl;
          s_victim_key[r] = a.cache.slot_key[sl];
        } else {
          a.cache.order_out[r - nM] = sl;
        }
        ++r;
      }
    }
    __syncthreads();
  }
  if (w != 0) return;
  // warp 0, lane u: distinct expert u of the call
  const int u = lane;
  int e = -1, key = -1, slot = -1, hit = 0, evicted = -1;
  if (u < nU) {
    e = s_uexp[u];
    key = a.layer * E + e;
    slot = s_uslot[u];
    hit = lru ? slot >= 0 : 1;
  }
  const int hrank = __popc(__ballot_sync(0xffffffffu, u < nU && hit) & lanemask_lt());
  const int mrank = u - hrank;
  if (lru && u < nU) {
    if (hit) {
      a.cache.order_out[S - nH - nM + hrank] = slot;
    } else {
      const int v = s_victim[mrank];
      a.cache.order_out[S - nM + mrank] = v;
      const int ek = s_victim_key[mrank];
      if (ek >= 0) {
        a.cache.key_slot[ek] = -1;
        evicted = ek;
      }
      a.cache.slot_key[v] = key;
      a.cache.key_slot[key] = v;
      slot = v;
    }
  }
  const int nEv = __popc(__ballot_sync(0xffffffffu, evicted >= 0));
  if (u < nU) {
    a.plan.u_expert[u] = e;
    a.plan.u_slot[u] = slot;
    a.plan.u_hit[u] = hit;
    a.plan.u_evicted[u] = evicted;
    a.plan.u_info[hit ? hrank : nH + mrank] = make_int4(e, slot, s_off[e], (s_count[e] << 1) | hit);
    if (!hit) {
      a.plan.miss[mrank] = make_int2(key, slot);
      if (a.mirror) {
        a.mirror[2 + mrank] = key;
        a.mirror[2 + a.umax + mrank] = slot;
      }
    }
  }
  __syncwarp();
  if (lane == 0) {
    if (a.mirror) {
      // the warp's miss-list writes precede this fence, and the host reads
      // the list only after it sees the new sequence number
      a.mirror[1] = nM;
      __threadfence_system();
      *(volatile int32_t *)&a.mirror[0] = (int32_t)a.seq;
    }
    a.plan.n[0] = nU;
    a.plan.n[1] = nH;
    a.plan.n[2] = nM;
    a.plan.n[3] = nEv;
    unsigned long long *st = a.cache.stats;
    const unsigned long long bytes = lru ? (unsigned long long)nM * a.blob_bytes : 0ull;
    const unsigned long long hits_ = lru ? nH : 0, miss_ = lru ? nM : 0;
    st[0] = pf.st[0] + nU; st[1] = pf.st[1] + hits_; st[2] = pf.st[2] + miss_; st[3] = pf.st[3] + nEv;
    st[4] = pf.st[4] + bytes;
    st[8] = nU; st[9] = hits_; st[10] = miss_; st[11] = nEv; st[12] = bytes;
  }
}

// Single-CTA routing: the decode-sized path when the call has at most 32
// (token, rank) pairs, else the general one.
__device__ __forceinline__ void route_body(const RouteArgs &a, int *smem, bool pdl) {
  if (a.T * a.k <= kDecodeRoutePairs) route_decode_body(a, smem, pdl);
  else route_small_body(a, smem, pdl);
}

}  // namespace
}  // namespace ftmoe
