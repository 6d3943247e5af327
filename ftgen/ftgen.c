/*
 * ftgen.c -- seeded synthetic inputs for the host-resident-expert MoE layer.
 *
 * This module only PRODUCES inputs: random numbers, and the packing of fp32
 * master weights into the expert blob formats.  It holds none of the layer's
 * own arithmetic (no routing, no cache policy, no decoding, no FFN).  Both the
 * CPU oracle and the GPU library consume the bytes written here; neither
 * links this file into its own computation.
 *
 * Random numbers: a counter-addressed SplitMix64 stream (Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014).  The i-th
 * output of a SplitMix64 generator whose state starts at k is
 * mix64(k + (i+1)*GAMMA); any element can therefore be drawn on its own.
 * Normal deviates use the Box-Muller transform (Box & Muller 1958) on pairs of
 * uniforms (element 2j takes the cosine branch, 2j+1 the sine branch).
 *
 * Blob formats (per expert, three matrices gate[I][H], up[I][H], down[H][I],
 * row-major, K contiguous; gate and up stacked as W_gu[2I][H]):
 *   BF16 : W_gu bf16[2I][H] | W_d bf16[H][I]                  -> 6*H*I bytes
 *   NVFP4: gu_codes u8[2I][H/2] | gu_sf e4m3[2I][H/16]
 *        | d_codes u8[H][I/2]   | d_sf e4m3[H][I/16]
 *        | f32 global scale[4] = {gate, up, down, 0}           -> 27*H*I/16 + 16
 *   MXFP4: gu_codes u8[2I][H/2] | gu_sf e8m0[2I][H/32]
 *        | d_codes u8[H][I/2]   | d_sf e8m0[H][I/32]           -> 51*H*I/32
 * FP4 codes: element 2j of a row in the low nibble of byte j, element 2j+1 in
 * the high nibble; bit 3 of a nibble is the sign.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* State of the stream (seed, stream): two finaliser rounds of the pair. */
static inline uint64_t stream_state(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed + GAMMA) + stream * GAMMA);
}

static inline uint64_t draw_u64(uint64_t state, uint64_t ctr) {
  return mix64(state + (ctr + 1) * GAMMA);
}

/* Uniform in [0, 1) with 24 random bits. */
static inline float draw_unit(uint64_t state, uint64_t ctr) {
  return (float)(draw_u64(state, ctr) >> 40) * (1.0f / 16777216.0f);
}

static inline float draw_normal(uint64_t state, uint64_t i) {
  uint64_t j = i >> 1;
  float u1 = draw_unit(state, 2 * j);
  float u2 = draw_unit(state, 2 * j + 1);
  float r = sqrtf(-2.0f * logf(1.0f - u1));
  float th = 6.283185307179586f * u2;
  return (i & 1) ? r * sinf(th) : r * cosf(th);
}

uint64_t ftgen_u64(uint64_t seed, uint64_t stream, uint64_t ctr) {
  return draw_u64(stream_state(seed, stream), ctr);
}

void ftgen_normal_f32(uint64_t seed, uint64_t stream, uint64_t ctr0, int64_t n, float *out) {
  uint64_t st = stream_state(seed, stream);
  for (int64_t i = 0; i < n; ++i) out[i] = draw_normal(st, ctr0 + (uint64_t)i);
}

void ftgen_uniform_f32(uint64_t seed, uint64_t stream, uint64_t ctr0, int64_t n, float *out) {
  uint64_t st = stream_state(seed, stream);
  for (int64_t i = 0; i < n; ++i) out[i] = draw_unit(st, ctr0 + (uint64_t)i);
}

/* Fisher-Yates shuffle of 0..n-1 driven by the stream (Durstenfeld order). */
void ftgen_permutation(uint64_t seed, uint64_t stream, int32_t n, int32_t *out) {
  uint64_t st = stream_state(seed, stream);
  for (int32_t i = 0; i < n; ++i) out[i] = i;
  for (int32_t i = n - 1; i > 0; --i) {
    uint64_t r = draw_u64(st, (uint64_t)i);
    int32_t j = (int32_t)(r % (uint64_t)(i + 1));
    int32_t t = out[i]; out[i] = out[j]; out[j] = t;
  }
}

/* ---------------- encoders (producer side of the formats) ---------------- */

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u; memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Nearest point of the e2m1 grid {0,.5,1,1.5,2,3,4,6}, ties to the even code,
 * magnitudes above 6 saturate.  Returns the 4-bit code. */
static uint8_t enc_e2m1(float v) {
  float a = fabsf(v);
  /* count the decision boundaries below a; "<" vs "<=" puts each tie on the
   * even code (0.25->0, 0.75->2, 1.25->2, 1.75->4, 2.5->4, 3.5->6, 5->6) */
  uint8_t c = (uint8_t)((a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) +
                        (a > 2.5f) + (a >= 3.5f) + (a > 5.0f));
  if (c != 0 && v < 0) c |= 8;
  return c;
}

/* Non-negative finite E4M3 (OCP "FN") values, codes 0..126. */
static float e4m3_pos[127];
static pthread_once_t e4m3_once = PTHREAD_ONCE_INIT;
static void e4m3_init(void) {
  for (int c = 0; c < 127; ++c) {
    int e = c >> 3, m = c & 7;
    e4m3_pos[c] = e ? ldexpf(1.0f + m / 8.0f, e - 7) : ldexpf(m / 8.0f, -6);
  }
}

/* Nearest non-negative E4M3 value to s >= 0, ties to the even code,
 * saturating at 448. */
static uint8_t enc_e4m3_pos(float s) {
  pthread_once(&e4m3_once, e4m3_init);
  if (!(s > 0.0f)) return 0;
  if (s >= 448.0f) return 126;
  int lo = 0, hi = 126; /* e4m3_pos[lo] <= s < e4m3_pos[hi] */
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (e4m3_pos[mid] <= s) lo = mid; else hi = mid;
  }
  float dl = s - e4m3_pos[lo], dh = e4m3_pos[hi] - s;
  if (dl < dh) return (uint8_t)lo;
  if (dh < dl) return (uint8_t)hi;
  return (uint8_t)((lo & 1) ? hi : lo);
}

static float e4m3_value(uint8_t c) {
  pthread_once(&e4m3_once, e4m3_init);
  return e4m3_pos[c & 127];
}

enum { FMT_BF16 = 0, FMT_NVFP4 = 1, FMT_MXFP4 = 2, FMT_FP8 = 3 };
enum { FLAG_NVFP4_UNIT_GSCALE = 1 };

int64_t ftgen_blob_bytes(int fmt, int64_t H, int64_t I) {
  switch (fmt) {
    case FMT_BF16: return 6 * H * I;
    case FMT_NVFP4: return 27 * H * I / 16 + 16;
    case FMT_MXFP4: return 51 * H * I / 32;
    case FMT_FP8: return 3 * H * I + 4 * (2 * I + H);
  }
  return -1;
}

/* Packs one matrix w[rows][K] into E4M3 codes[rows][K] (sign in bit 7) and one
 * fp32 scale per row: scale = absmax(row) / 448, code = nearest E4M3 of
 * w / scale (ties to even, saturating at 448). */
static void pack_fp8(const float *w, int64_t rows, int64_t K, uint8_t *codes, float *scale) {
  for (int64_t r = 0; r < rows; ++r) {
    const float *wr = w + r * K;
    float amax = 0.0f;
    for (int64_t i = 0; i < K; ++i) amax = fmaxf(amax, fabsf(wr[i]));
    float sc = amax / 448.0f;
    if (!(sc > 0.0f)) sc = 1.0f;
    scale[r] = sc;
    for (int64_t i = 0; i < K; ++i) {
      const float v = wr[i] / sc;
      uint8_t c = enc_e4m3_pos(fabsf(v));
      if (v < 0 && c != 0) c |= 0x80;
      codes[r * K + i] = c;
    }
  }
}

/* Packs one matrix w[rows][K] into codes[rows][K/2] and scale bytes. */
static void pack_nvfp4(const float *w, int64_t rows, int64_t K, float g,
                       uint8_t *codes, uint8_t *sf) {
  for (int64_t r = 0; r < rows; ++r) {
    const float *wr = w + r * K;
    for (int64_t b = 0; b < K / 16; ++b) {
      float amax = 0.0f;
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(wr[b * 16 + i]));
      uint8_t sc = enc_e4m3_pos(amax / (6.0f * g));
      sf[r * (K / 16) + b] = sc;
      float step = e4m3_value(sc) * g;
      for (int i = 0; i < 16; i += 2) {
        uint8_t lo = step > 0 ? enc_e2m1(wr[b * 16 + i] / step) : 0;
        uint8_t hi = step > 0 ? enc_e2m1(wr[b * 16 + i + 1] / step) : 0;
        codes[r * (K / 2) + b * 8 + i / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
}

static void pack_mxfp4(const float *w, int64_t rows, int64_t K, uint8_t *codes, uint8_t *sf) {
  for (int64_t r = 0; r < rows; ++r) {
    const float *wr = w + r * K;
    for (int64_t b = 0; b < K / 32; ++b) {
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(wr[b * 32 + i]));
      int e;
      if (amax > 0.0f) {
        int ex; frexpf(amax, &ex);           /* amax = f * 2^ex, f in [0.5,1) */
        e = (ex - 1) - 2;                     /* floor(log2 amax) - emax(e2m1) */
        if (e < -127) e = -127;
        if (e > 127) e = 127;
      } else {
        e = -127;
      }
      sf[r * (K / 32) + b] = (uint8_t)(e + 127);
      float step = ldexpf(1.0f, e);
      for (int i = 0; i < 32; i += 2) {
        uint8_t lo = amax > 0 ? enc_e2m1(wr[b * 32 + i] / step) : 0;
        uint8_t hi = amax > 0 ? enc_e2m1(wr[b * 32 + i + 1] / step) : 0;
        codes[r * (K / 2) + b * 16 + i / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
}

/* Fills w[n] with wstd * N(0,1) drawn at counters ctr0..ctr0+n-1 of the expert's stream. */
static void master(uint64_t st, uint64_t ctr0, int64_t n, float wstd, float *w) {
  int64_t i = 0;
  if (ctr0 & 1) { w[0] = wstd * draw_normal(st, ctr0); i = 1; }
  for (; i + 1 < n; i += 2) {  /* one Box-Muller pair per two elements */
    uint64_t j = (ctr0 + (uint64_t)i) >> 1;
    float u1 = draw_unit(st, 2 * j), u2 = draw_unit(st, 2 * j + 1);
    float r = wstd * sqrtf(-2.0f * logf(1.0f - u1));
    float sn, cs;
    sincosf(6.283185307179586f * u2, &sn, &cs);
    w[i] = r * cs;
    w[i + 1] = r * sn;
  }
  if (i < n) w[i] = wstd * draw_normal(st, ctr0 + (uint64_t)i);
}

static float absmax(const float *w, int64_t n) {
  float a = 0.0f;
  for (int64_t i = 0; i < n; ++i) a = fmaxf(a, fabsf(w[i]));
  return a;
}

/* One expert blob for logical key `key`.  tmp holds max(I*H) floats. */
static void expert_blob(int fmt, int64_t H, int64_t I, float wstd, uint64_t seed,
                        uint64_t key, int flags, uint8_t *out, float *tmp) {
  uint64_t st = stream_state(seed, 0x4558505254000000ULL + key); /* "EXPRT" + key */
  const int64_t HI = H * I;
  if (fmt == FMT_BF16) {
    uint16_t *gu = (uint16_t *)out, *d = gu + 2 * HI;
    for (int m = 0; m < 3; ++m) {
      master(st, (uint64_t)(m * HI), HI, wstd, tmp);
      uint16_t *dst = m == 0 ? gu : (m == 1 ? gu + HI : d);
      for (int64_t i = 0; i < HI; ++i) dst[i] = f32_to_bf16_rne(tmp[i]);
    }
  } else if (fmt == FMT_NVFP4) {
    uint8_t *gu_c = out, *gu_s = gu_c + HI, *d_c = gu_s + HI / 8, *d_s = d_c + HI / 2;
    float *gs = (float *)(d_s + HI / 16);
    for (int m = 0; m < 3; ++m) {
      master(st, (uint64_t)(m * HI), HI, wstd, tmp);
      float g = (flags & FLAG_NVFP4_UNIT_GSCALE) ? 1.0f : absmax(tmp, HI) / (6.0f * 448.0f);
      if (!(g > 0.0f)) g = 1.0f;
      gs[m] = g;
      if (m < 2) pack_nvfp4(tmp, I, H, g, gu_c + m * (HI / 2), gu_s + m * (HI / 16));
      else pack_nvfp4(tmp, H, I, g, d_c, d_s);
    }
    gs[3] = 0.0f;
  } else if (fmt == FMT_FP8) {
    /* gu codes [2I][H] | gu scales f32 [2I] | d codes [H][I] | d scales f32 [H] */
    uint8_t *gu_c = out;
    float *gu_s = (float *)(gu_c + 2 * HI);
    uint8_t *d_c = (uint8_t *)(gu_s + 2 * I);
    float *d_s = (float *)(d_c + HI);
    for (int m = 0; m < 3; ++m) {
      master(st, (uint64_t)(m * HI), HI, wstd, tmp);
      if (m < 2) pack_fp8(tmp, I, H, gu_c + m * HI, gu_s + m * I);
      else pack_fp8(tmp, H, I, d_c, d_s);
    }
  } else {
    uint8_t *gu_c = out, *gu_s = gu_c + HI, *d_c = gu_s + HI / 16, *d_s = d_c + HI / 2;
    for (int m = 0; m < 3; ++m) {
      master(st, (uint64_t)(m * HI), HI, wstd, tmp);
      if (m < 2) pack_mxfp4(tmp, I, H, gu_c + m * (HI / 2), gu_s + m * (HI / 32));
      else pack_mxfp4(tmp, H, I, d_c, d_s);
    }
  }
}

/* fp32 master weights of one expert (gate[I][H], up[I][H], down[H][I]) --
 * the values the blob encodes before quantisation. */
void ftgen_master_weights(int64_t H, int64_t I, float wstd, uint64_t seed, uint64_t key,
                          float *gate, float *up, float *down) {
  uint64_t st = stream_state(seed, 0x4558505254000000ULL + key);
  const int64_t HI = H * I;
  master(st, 0, HI, wstd, gate);
  master(st, (uint64_t)HI, HI, wstd, up);
  master(st, (uint64_t)(2 * HI), HI, wstd, down);
}

typedef struct {
  int fmt, flags, tid, nthreads;
  int64_t H, I, n, stride;
  float wstd;
  uint64_t seed;
  const uint64_t *keys;
  uint8_t *out;
  int rc;
} job_t;

static void *pool_worker(void *arg) {
  job_t *j = (job_t *)arg;
  float *tmp = (float *)malloc(sizeof(float) * (size_t)(j->H * j->I));
  if (!tmp) { j->rc = -1; return NULL; }
  for (int64_t i = j->tid; i < j->n; i += j->nthreads)
    expert_blob(j->fmt, j->H, j->I, j->wstd, j->seed, j->keys[i], j->flags,
                j->out + i * j->stride, tmp);
  free(tmp);
  j->rc = 0;
  return NULL;
}

/* Writes n blobs (keys[i]) at out + i*stride, using nthreads threads. */
int ftgen_pool(int fmt, int64_t H, int64_t I, float wstd, uint64_t seed, int flags,
               const uint64_t *keys, int64_t n, uint8_t *out, int64_t stride, int nthreads) {
  if (ftgen_blob_bytes(fmt, H, I) < 0 || stride < ftgen_blob_bytes(fmt, H, I)) return -1;
  if (H % 32 || I % 32) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  job_t jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (job_t){fmt, flags, t, nthreads, H, I, n, stride, wstd, seed, keys, out, -1};
    if (pthread_create(&th[t], NULL, pool_worker, &jobs[t]) != 0) { nthreads = t; break; }
  }
  int rc = nthreads > 0 ? 0 : -1;
  for (int t = 0; t < nthreads; ++t) {
    pthread_join(th[t], NULL);
    if (jobs[t].rc) rc = -1;
  }
  return rc;
}

/* f32 -> bf16 bits with round-to-nearest-even (inputs are finite). */
void ftgen_to_bf16(const float *in, int64_t n, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}
