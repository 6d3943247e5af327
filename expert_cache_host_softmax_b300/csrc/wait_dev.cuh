// wait_dev.cuh -- bounded device-side waits and the miss-copy loop, shared by
// the GEMV kernels, the miss-copy kernel and the fused decode layer kernel.
//
// Every wait gives up after kWaitNs of the global timer: it records its site
// in the device error word (the host reports FT_ERR_DEVICE at its next
// synchronising call) and the CTA skips the work that needed the wait.
#pragma once
#include "ft_internal.cuh"

namespace ftmoe {
namespace {

constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s per wait

__device__ __forceinline__ unsigned long long dev_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Thread 0 waits until *flag == want (bounded); the whole CTA learns the
// outcome.  The CTA's later reads see what was written before the flag.
__device__ __forceinline__ bool cta_wait_flag(const int *flag, int want, int *err, int site, int *s_ok) {
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
        __nanosleep(64);
      }
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Copies ranges [s0, s1) of a.seg of every miss of the call from its pinned
// host blob into its slot.  Thread `t` of `nt` copying threads takes slots
// t, t + nt, ... of a padded word index: each miss's range gets a multiple of
// 8 sixteen-byte slots, shifted so that slot 0 sits on a 128-byte boundary of
// the host address.  A warp thus reads whole, aligned 128-byte lines over
// PCIe (the pool's blobs need only be 16-byte aligned); slots outside the
// range copy nothing.
constexpr int kCopyUnroll = 4;   // 16-byte loads in flight per thread and round
__device__ __forceinline__ void copy_misses(const MissCopyArgs &a, int s0, int s1, long long t, long long nt) {
  const int n_miss = a.n[2];
  for (int sg = s0; sg < s1; ++sg) {
    const long long per = (a.seg[sg][1] - a.seg[sg][0]) >> 4;
    if (per == 0) continue;
    const long long per_pad = (per + 7 + 7) & ~7ll;
    const long long total = per_pad * n_miss;
    for (long long base = t; base < total; base += nt * kCopyUnroll) {
      uint4 v[kCopyUnroll];
      uint4 *dst[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const long long w = base + u * nt;
        dst[u] = nullptr;
        if (w < total) {
          const int i = (int)(w / per_pad);
          const int2 m = a.miss[i];
          const uint8_t *src0 = reinterpret_cast<const uint8_t *>(a.pool_dev[m.x]) + a.seg[sg][0];
          const long long word = (w - (long long)i * per_pad) - (long long)((reinterpret_cast<uintptr_t>(src0) >> 4) & 7);
          if (word >= 0 && word < per) {
            dst[u] = reinterpret_cast<uint4 *>(a.slots + (size_t)m.y * a.slot_stride + a.seg[sg][0] + (word << 4));
            v[u] = __ldg(reinterpret_cast<const uint4 *>(src0) + word);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u)
        if (dst[u]) *dst[u] = v[u];
    }
  }
}

// The last of `n_ctas` CTAs to arrive sets *flag = value (after every CTA's
// earlier writes) and re-arms the counter.
__device__ __forceinline__ void cta_arrive_last_sets(int *count, int *flag, int n_ctas, int value) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(count, 1) == n_ctas - 1) {
    *count = 0;
    __threadfence();
    atomicExch(flag, value);
  }
}

}  // namespace
}  // namespace ftmoe
