/*
 * synth.c — seeded synthetic inputs shared by the GPU path's harness and the
 * oracle's tests.  It draws numbers and nothing else: no quantisation, no
 * linear algebra, no part of the decode method lives here.
 *
 * Generator (counter based, so every element is a pure function of
 * (seed, tensor id, element index) and the thread split cannot change it):
 *   mix(z)      = the SplitMix64 output finaliser (Steele, Lea & Flood,
 *                 "Fast splittable pseudorandom number generators", 2014):
 *                 z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                 z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   key(s, t)   = mix(s + GOLDEN * (mix(t + 0x632BE59BD9B4E019) | 1))
 *   r(s, t, j)  = mix(key(s, t) + (j + 1) * GOLDEN),  GOLDEN = 0x9E3779B97F4A7C15
 * Normal draws use the Box–Muller transform on pair j = i/2:
 *   u1 = ((r >> 40) + 0.5) / 2^24,  u2 = ((r >> 16) & 0xFFFFFF) / 2^24
 *   z_even = sqrt(-2 ln u1) cos(2 pi u2),  z_odd = sqrt(-2 ln u1) sin(2 pi u2)
 * and the value mu + sigma * z is rounded double -> fp32 -> bf16, each step
 * round-to-nearest-even.  Integer draws take the top 32 bits of r(s, t, i) and
 * map them onto [0, n) by a 32x32 -> 64 bit multiply-shift.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27; z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return mix64(seed + GOLDEN * (mix64(tid + 0x632BE59BD9B4E019ULL) | 1ULL));
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u; memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

uint64_t synth_raw(uint64_t seed, uint64_t tid, uint64_t j) {
  return mix64(stream_key(seed, tid) + (j + 1) * GOLDEN);
}

static double normal_at(uint64_t key, uint64_t i) {
  uint64_t r = mix64(key + ((i >> 1) + 1) * GOLDEN);
  double u1 = ((double)(r >> 40) + 0.5) * (1.0 / 16777216.0);
  double u2 = (double)((r >> 16) & 0xFFFFFFu) * (1.0 / 16777216.0);
  double rad = sqrt(-2.0 * log(u1));
  double ang = 6.283185307179586 * u2;
  return (i & 1) ? rad * sin(ang) : rad * cos(ang);
}

typedef struct {
  uint64_t key, i0, i1;
  double mu, sigma;
  uint16_t* out_bf16;
  float* out_f32;
} job_t;

static void* normal_worker(void* p) {
  job_t* j = (job_t*)p;
  for (uint64_t i = j->i0; i < j->i1; ++i) {
    float v = (float)(j->mu + j->sigma * normal_at(j->key, i));
    if (j->out_bf16) j->out_bf16[i] = f32_to_bf16_rne(v);
    else j->out_f32[i] = v;
  }
  return 0;
}

static void run_normal(uint64_t seed, uint64_t tid, uint64_t n, double mu, double sigma,
                       uint16_t* ob, float* of, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (n < (1u << 16)) nthreads = 1;
  uint64_t key = stream_key(seed, tid);
  pthread_t th[64];
  job_t jobs[64];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].key = key; jobs[t].mu = mu; jobs[t].sigma = sigma;
    jobs[t].i0 = n * (uint64_t)t / (uint64_t)nthreads;
    jobs[t].i1 = n * (uint64_t)(t + 1) / (uint64_t)nthreads;
    jobs[t].out_bf16 = ob; jobs[t].out_f32 = of;
  }
  if (nthreads == 1) { normal_worker(&jobs[0]); return; }
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], 0, normal_worker, &jobs[t]);
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], 0);
}

/* n bf16 values ~ mu + sigma * N(0,1) for tensor `tid`, element i at out[i]. */
void synth_normal_bf16(uint64_t seed, uint64_t tid, uint64_t n, double mu, double sigma,
                       uint16_t* out, int nthreads) {
  run_normal(seed, tid, n, mu, sigma, out, 0, nthreads);
}

/* Same draws kept at fp32 (no bf16 rounding). */
void synth_normal_f32(uint64_t seed, uint64_t tid, uint64_t n, double mu, double sigma,
                      float* out, int nthreads) {
  run_normal(seed, tid, n, mu, sigma, 0, out, nthreads);
}

/* n integers uniform on [0, range). */
void synth_uniform_int(uint64_t seed, uint64_t tid, uint64_t n, uint32_t range, int32_t* out) {
  uint64_t key = stream_key(seed, tid);
  for (uint64_t i = 0; i < n; ++i) {
    uint64_t r = mix64(key + (i + 1) * GOLDEN);
    out[i] = (int32_t)(((r >> 32) * (uint64_t)range) >> 32);
  }
}
