/*
 * synth.c -- seeded, counter-based synthetic input generator.
 *
 * This file produces the raw random draws that both the CPU oracle and the
 * CUDA path consume.  It contains none of the attention method's arithmetic:
 * no scores, no selection, no softmax.  Every value is a pure function of
 * (key, element index), so the result does not depend on the thread count.
 *
 * Generator definitions (all published, restated here):
 *   - SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014): state advances by the golden gamma
 *     0x9E3779B97F4A7C15 and each output is passed through the mix function
 *     z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27; z *= 0x94D049BB133111EB;
 *     z ^= z>>31.  Used here in counter mode: draw(key, i) = mix(key + (i+1)*gamma).
 *   - Uniform on (0,1): ((x >> 11) + 0.5) * 2^-53.
 *   - Box-Muller (Box and Muller 1958), cosine branch only:
 *     N = sqrt(-2 ln u1) * cos(2 pi u2), u1 = U(draw 2i), u2 = U(draw 2i+1),
 *     evaluated in double, then rounded to float.
 *   - float -> bfloat16 by round-to-nearest-even on the upper 16 bits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t syn_mix(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t syn_draw(uint64_t key, uint64_t i) {
  return syn_mix(key + (i + 1) * SYN_GAMMA);
}

static inline double syn_unit(uint64_t x) {
  return ((double)(x >> 11) + 0.5) * 0x1.0p-53;
}

static inline double syn_normal_at(uint64_t key, uint64_t i) {
  double u1 = syn_unit(syn_draw(key, 2 * i));
  double u2 = syn_unit(syn_draw(key, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

static inline uint16_t syn_f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) { /* inf / nan: keep, quiet nans */
    uint16_t h = (uint16_t)(u >> 16);
    if (u & 0x007FFFFFu) h |= 0x0040u;
    return h;
  }
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* Derive a stream key from a seed and up to three small integers. */
uint64_t syn_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b) {
  uint64_t z = syn_mix(seed * SYN_GAMMA + 0x1234567ULL);
  z = syn_mix(z ^ (tag * 0xD1B54A32D192ED03ULL));
  z = syn_mix(z ^ (a * 0x8CB92BA72F3D8DD7ULL));
  z = syn_mix(z ^ (b * 0xABC98388FB8FAC03ULL));
  return z;
}

uint64_t syn_u64(uint64_t key, uint64_t i) { return syn_draw(key, i); }

double syn_normal1(uint64_t key, uint64_t i) { return syn_normal_at(key, i); }

typedef struct {
  uint64_t key;
  uint64_t first;   /* counter of dst[0] */
  int64_t count;
  int dtype;        /* 0: float32, 1: bfloat16 bits, 2: float64 */
  double mean, std; /* value = mean + std * N */
  void *dst;
  int nthreads;
  int tid;
} syn_job;

static void *syn_worker(void *arg) {
  syn_job *j = (syn_job *)arg;
  int64_t per = (j->count + j->nthreads - 1) / j->nthreads;
  int64_t lo = per * j->tid, hi = lo + per;
  if (hi > j->count) hi = j->count;
  for (int64_t e = lo; e < hi; ++e) {
    double x = j->mean + j->std * syn_normal_at(j->key, j->first + (uint64_t)e);
    float f = (float)x;
    if (j->dtype == 2)
      ((double *)j->dst)[e] = x;
    else if (j->dtype == 0)
      ((float *)j->dst)[e] = f;
    else
      ((uint16_t *)j->dst)[e] = syn_f32_to_bf16_bits(f);
  }
  return NULL;
}

/* dst[e] = round_dtype(mean + std * N(key, first + e)), e in [0, count). */
void syn_fill_normal(uint64_t key, uint64_t first, int64_t count, int dtype,
                     double mean, double std, void *dst, int nthreads) {
  if (count <= 0) return;
  if (nthreads < 1) nthreads = 1;
  if (count < (1 << 16)) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  syn_job jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (syn_job){key, first, count, dtype, mean, std, dst, nthreads, t};
    if (nthreads == 1) {
      syn_worker(&jobs[t]);
    } else if (pthread_create(&th[t], NULL, syn_worker, &jobs[t]) != 0) {
      syn_worker(&jobs[t]);
      th[t] = 0;
    }
  }
  if (nthreads > 1)
    for (int t = 0; t < nthreads; ++t)
      if (th[t]) pthread_join(th[t], NULL);
}

/* Round float32 values to bfloat16 bits (round-to-nearest-even). */
void syn_f32_to_bf16(const float *src, uint16_t *dst, int64_t count) {
  for (int64_t e = 0; e < count; ++e) dst[e] = syn_f32_to_bf16_bits(src[e]);
}
