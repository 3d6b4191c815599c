/*
 * synth.c -- seeded counter-based generator for synthetic W4A16 inputs.
 *
 * The definitions of every draw are in include/w4a16_synth.h.  This file only
 * draws numbers and stores them in the packed format; it computes nothing of
 * the quantized matmul itself.  Work is split over host threads in fixed,
 * index-addressed chunks, so results do not depend on the thread count.
 *
 * The input distributions follow the workloads the pages describe: bf16
 * activations, unsigned 4-bit codes packed eight to a uint32 low nibble first
 * (tiny-llm "Week 2 Day 2: Keep W4 Packed", section "Packed Storage Layout"),
 * and one bf16 scale and bias per 64-column group (group size 64, from the
 * "Gemma 4 E4B & E2B -- single-launch Metal megakernels" model card, section
 * "Usage").  Scales are kept finite and positive-range, as the "Hy4-preview
 * Metal kernels for llama.cpp" notes ("Test-data hygiene") advise.
 *
 * The same page's STQ1_0 blocks (section "Notes and gotchas": 32 bytes of
 * 4-bit group codes, 8 bytes of group sign bits, an fp16 scale; 42 bytes per
 * 256 weights) are drawn as uniform random bytes and a finite fp16 scale,
 * with float32 activations for its _f32 kernels.
 */
#include "w4a16_synth.h"

#include <math.h>
#include <pthread.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL
#define TID_SPREAD 0xD1B54A32D192ED03ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint32_t tid) {
  return mix64(seed ^ ((uint64_t)tid * TID_SPREAD));
}

static inline uint64_t hash_at(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * GOLDEN_GAMMA);
}

/* IEEE-754 binary32 -> bfloat16, round to nearest, ties to even; NaN stays a
 * quiet NaN with its sign. */
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* IEEE-754 binary32 -> binary16, round to nearest, ties to even, through
 * exact double arithmetic: v = r * spacing with r rounded to an integer. */
static uint16_t f32_to_fp16(float f) {
  const uint16_t sign = signbit(f) ? 0x8000 : 0;
  if (isnan(f)) return (uint16_t)(sign | 0x7E00);
  double a = fabs((double)f);
  if (isinf(a)) return (uint16_t)(sign | 0x7C00);
  if (a == 0.0) return sign;
  int ex;
  frexp(a, &ex); /* a = m * 2^ex, m in [0.5, 1): binade exponent ex - 1 */
  int e = ex - 1;
  int spacing_exp = (e < -14) ? -24 : e - 10;
  double q = ldexp(a, -spacing_exp), fl = floor(q), diff = q - fl, r;
  if (diff > 0.5) r = fl + 1.0;
  else if (diff < 0.5) r = fl;
  else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  double res = ldexp(r, spacing_exp);
  if (res >= 65520.0) return (uint16_t)(sign | 0x7C00);
  if (res < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)r); /* subnormal or 2^-14 itself */
  frexp(res, &ex);
  e = ex - 1;
  double sig = ldexp(res, -(e - 10)); /* in [1024, 2048) */
  return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)sig - 1024));
}

static inline double uniform24(uint64_t h) { return (double)(h >> 40) * (1.0 / 16777216.0); }

static inline double normal_at(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t h1 = hash_at(key, 2 * i), h2 = hash_at(key, 2 * i + 1);
  double u1 = ((double)(h1 >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0,1] */
  double u2 = (double)(h2 >> 11) * (1.0 / 9007199254740992.0);         /* [0,1) */
  return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

/* ---- fixed-chunk parallel-for over [0, n) --------------------------------- */

typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);

typedef struct {
  range_fn fn;
  void* ctx;
  int64_t n, chunk;
  int nthreads, me;
} job_t;

static void* job_run(void* p) {
  job_t* j = (job_t*)p;
  for (int64_t c = j->me; c * j->chunk < j->n; c += j->nthreads) {
    int64_t lo = c * j->chunk, hi = lo + j->chunk;
    if (hi > j->n) hi = j->n;
    j->fn(j->ctx, lo, hi);
  }
  return NULL;
}

int w4a16_synth_threads(void) {
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  if (c < 1) c = 1;
  if (c > 64) c = 64;
  return (int)c;
}

static void parallel_for(int64_t n, range_fn fn, void* ctx) {
  const int64_t chunk = 1 << 16;
  int nt = w4a16_synth_threads();
  if (n <= chunk || nt == 1) {
    if (n > 0) fn(ctx, 0, n);
    return;
  }
  if ((int64_t)nt > (n + chunk - 1) / chunk) nt = (int)((n + chunk - 1) / chunk);
  pthread_t th[64];
  job_t jobs[64];
  int started[64];
  for (int t = 0; t < nt; ++t) {
    jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].n = n; jobs[t].chunk = chunk;
    jobs[t].nthreads = nt; jobs[t].me = t;
    started[t] = (t > 0) && pthread_create(&th[t], NULL, job_run, &jobs[t]) == 0;
  }
  job_run(&jobs[0]);
  for (int t = 1; t < nt; ++t) {
    if (started[t]) pthread_join(th[t], NULL);
    else job_run(&jobs[t]); /* thread creation failed: run the share inline */
  }
}

/* ---- tensors ---------------------------------------------------------------- */

typedef struct { uint64_t key, offset; void* out; void* out2; uint64_t key2; } ctx_t;

static void do_hash(void* p, int64_t lo, int64_t hi) {
  ctx_t* c = (ctx_t*)p;
  uint64_t* o = (uint64_t*)c->out;
  for (int64_t i = lo; i < hi; ++i) o[i] = hash_at(c->key, c->offset + (uint64_t)i);
}

int w4a16_synth_hash(uint64_t seed, uint32_t tid, uint64_t offset, int64_t n, uint64_t* out) {
  if (n < 0) return -2;
  if (n > 0 && !out) return -1;
  ctx_t c = {stream_key(seed, tid), offset, out, NULL, 0};
  parallel_for(n, do_hash, &c);
  return 0;
}

static void do_x(void* p, int64_t lo, int64_t hi) {
  ctx_t* c = (ctx_t*)p;
  uint16_t* o = (uint16_t*)c->out;
  for (int64_t i = lo; i < hi; ++i) o[i] = f32_to_bf16((float)normal_at(c->key, c->offset + (uint64_t)i));
}

int w4a16_synth_x(uint64_t seed, uint64_t offset, int64_t n, uint16_t* out) {
  if (n < 0) return -2;
  if (n > 0 && !out) return -1;
  ctx_t c = {stream_key(seed, W4A16_SYNTH_TID_X), offset, out, NULL, 0};
  parallel_for(n, do_x, &c);
  return 0;
}

static void do_codes(void* p, int64_t lo, int64_t hi) {
  ctx_t* c = (ctx_t*)p;
  uint32_t* o = (uint32_t*)c->out;
  for (int64_t i = lo; i < hi; ++i) o[i] = (uint32_t)(hash_at(c->key, c->offset + (uint64_t)i) >> 32);
}

int w4a16_synth_codes(uint64_t seed, uint64_t offset, int64_t n, uint32_t* out) {
  if (n < 0) return -2;
  if (n > 0 && !out) return -1;
  ctx_t c = {stream_key(seed, W4A16_SYNTH_TID_CODES), offset, out, NULL, 0};
  parallel_for(n, do_codes, &c);
  return 0;
}

static void do_params(void* p, int64_t lo, int64_t hi) {
  ctx_t* c = (ctx_t*)p;
  uint16_t* so = (uint16_t*)c->out;
  uint16_t* bo = (uint16_t*)c->out2;
  for (int64_t i = lo; i < hi; ++i) {
    uint64_t idx = c->offset + (uint64_t)i;
    float s = (float)(0.002 + 0.018 * uniform24(hash_at(c->key, idx)));
    uint16_t sb = f32_to_bf16(s);
    if (so) so[i] = sb;
    if (bo) {
      uint32_t su = (uint32_t)sb << 16;
      float sf;
      memcpy(&sf, &su, 4);
      double b = -8.0 * (double)sf + 1e-3 * normal_at(c->key2, idx);
      bo[i] = f32_to_bf16((float)b);
    }
  }
}

int w4a16_synth_group_params(uint64_t seed, uint64_t offset, int64_t n, uint16_t* scales, uint16_t* biases) {
  if (n < 0) return -2;
  if (n > 0 && !scales && !biases) return -1;
  ctx_t c = {stream_key(seed, W4A16_SYNTH_TID_SCALES), offset, scales, biases,
             stream_key(seed, W4A16_SYNTH_TID_BIAS_NOISE)};
  parallel_for(n, do_params, &c);
  return 0;
}

int w4a16_synth_ids(uint64_t seed, int64_t T, int32_t E, int32_t* out) {
  if (T < 0 || E <= 0) return -2;
  if (T > 0 && !out) return -1;
  uint64_t key = stream_key(seed, W4A16_SYNTH_TID_IDS);
  for (int64_t t = 0; t < T; ++t) {
    uint64_t h = hash_at(key, (uint64_t)t) >> 32;
    out[t] = (int32_t)((h * (uint64_t)E) >> 32);
  }
  return 0;
}

static void do_x_f32(void* p, int64_t lo, int64_t hi) {
  ctx_t* c = (ctx_t*)p;
  float* o = (float*)c->out;
  for (int64_t i = lo; i < hi; ++i) o[i] = (float)normal_at(c->key, c->offset + (uint64_t)i);
}

int w4a16_synth_x_f32(uint64_t seed, uint64_t offset, int64_t n, float* out) {
  if (n < 0) return -2;
  if (n > 0 && !out) return -1;
  ctx_t c = {stream_key(seed, W4A16_SYNTH_TID_X), offset, out, NULL, 0};
  parallel_for(n, do_x_f32, &c);
  return 0;
}

static void do_stq1(void* p, int64_t lo, int64_t hi) {
  ctx_t* c = (ctx_t*)p;
  uint8_t* o = (uint8_t*)c->out;
  for (int64_t i = lo; i < hi; ++i) {
    const uint64_t blk = c->offset + (uint64_t)i;
    uint8_t* b = o + i * 42;
    for (int w = 0; w < 5; ++w) { /* 40 bytes: qs[32] then sign[8] */
      const uint64_t h = hash_at(c->key, blk * 5 + (uint64_t)w);
      for (int j = 0; j < 8; ++j) b[w * 8 + j] = (uint8_t)(h >> (8 * j));
    }
    const uint16_t d = f32_to_fp16((float)(0.002 + 0.018 * uniform24(hash_at(c->key2, blk))));
    b[40] = (uint8_t)(d & 0xFF);
    b[41] = (uint8_t)(d >> 8);
  }
}

int w4a16_synth_stq1(uint64_t seed, uint64_t offset, int64_t n, uint8_t* out) {
  if (n < 0) return -2;
  if (n > 0 && !out) return -1;
  ctx_t c = {stream_key(seed, W4A16_SYNTH_TID_STQ1_BITS), offset, out, NULL,
             stream_key(seed, W4A16_SYNTH_TID_STQ1_SCALE)};
  parallel_for(n, do_stq1, &c);
  return 0;
}

int w4a16_synth_fp16(float v, uint16_t* out) {
  if (!out) return -1;
  *out = f32_to_fp16(v);
  return 0;
}
