/*
 * Seeded synthetic-input generator (host C, no GPU).
 *
 * This module produces the workload's inputs (weights, start ids, draft ids
 * and draft coins) from a seed.  It holds none of the verify step's
 * arithmetic: both the CUDA library and the fp64 oracle receive the arrays it
 * writes as plain inputs, so the two sides see identical values.
 *
 * Generator definition (counter based, so any element can be drawn on its
 * own and threads need no coordination):
 *   splitmix64(x): the 64-bit finaliser of Steele, Lea and Flood's SplitMix
 *     ("Fast splittable pseudorandom number generators", OOPSLA 2014) in the
 *     public-domain form Vigna gives: x += 0x9E3779B97F4A7C15, then two
 *     xor-shift-multiply rounds and a final xor-shift.
 *   draw(seed, tid, i) = splitmix64(splitmix64(splitmix64(seed) + tid) + i)
 *     tid names the tensor (or stream), i the element.
 *   uniform in [0,1):  (draw >> 11) * 2^-53
 *   normal pair j:     Box-Muller (Box and Muller, Ann. Math. Stat. 1958)
 *     u1 = ((draw(2j) >> 11) + 1) * 2^-53  in (0,1]
 *     u2 =  (draw(2j+1) >> 11) * 2^-53     in [0,1)
 *     element 2j   = sqrt(-2 ln u1) * cos(2 pi u2)
 *     element 2j+1 = sqrt(-2 ln u1) * sin(2 pi u2)
 *   bf16 weights: sigma * normal, rounded once from fp64 to bf16,
 *     round-to-nearest-even (overflow to infinity is impossible at the
 *     sigmas used).
 *   ids: draw % V.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_API __attribute__((visibility("default")))

static inline uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return splitmix64(splitmix64(seed) + tid);
}

static inline uint64_t draw_at(uint64_t key, uint64_t i) { return splitmix64(key + i); }

static const double kTwoPi = 6.283185307179586476925286766559;
static const double kInv53 = 1.0 / 9007199254740992.0; /* 2^-53 */

static inline double normal_at(uint64_t key, uint64_t i) {
  uint64_t j = i >> 1;
  double u1 = (double)((draw_at(key, 2 * j) >> 11) + 1) * kInv53;
  double u2 = (double)(draw_at(key, 2 * j + 1) >> 11) * kInv53;
  double r = sqrt(-2.0 * log(u1));
  return (i & 1) ? r * sin(kTwoPi * u2) : r * cos(kTwoPi * u2);
}

/* fp64 -> bf16 bits, round to nearest even (finite inputs of normal size). */
static inline uint16_t to_bf16(double x) {
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  int e = ilogb(x);
  if (e < -126) e = -126;
  double ulp = ldexp(1.0, e - 7);
  double y = rint(x / ulp) * ulp; /* exact: scaling by a power of two */
  float yf = (float)y;           /* exact: y has <= 8 significant bits */
  uint32_t bits;
  memcpy(&bits, &yf, 4);
  return (uint16_t)(bits >> 16);
}

typedef struct {
  int kind; /* 0 normal bf16, 1 ids, 2 uniform f64 */
  void* out;
  int64_t begin, end;
  uint64_t key, first;
  double sigma;
  int64_t modulus;
} job_t;

static void* run_job(void* p) {
  job_t* j = (job_t*)p;
  if (j->kind == 0) {
    /* Whole Box-Muller pairs are formed once and both halves kept. */
    uint16_t* o = (uint16_t*)j->out;
    int64_t i = j->begin;
    for (; i < j->end && ((j->first + (uint64_t)i) & 1); ++i)
      o[i] = to_bf16(j->sigma * normal_at(j->key, j->first + (uint64_t)i));
    for (; i + 1 < j->end; i += 2) {
      uint64_t pj = (j->first + (uint64_t)i) >> 1;
      double u1 = (double)((draw_at(j->key, 2 * pj) >> 11) + 1) * kInv53;
      double u2 = (double)(draw_at(j->key, 2 * pj + 1) >> 11) * kInv53;
      double r = sqrt(-2.0 * log(u1));
      o[i] = to_bf16(j->sigma * (r * cos(kTwoPi * u2)));
      o[i + 1] = to_bf16(j->sigma * (r * sin(kTwoPi * u2)));
    }
    for (; i < j->end; ++i)
      o[i] = to_bf16(j->sigma * normal_at(j->key, j->first + (uint64_t)i));
  } else if (j->kind == 1) {
    int32_t* o = (int32_t*)j->out;
    for (int64_t i = j->begin; i < j->end; ++i)
      o[i] = (int32_t)(draw_at(j->key, j->first + (uint64_t)i) % (uint64_t)j->modulus);
  } else {
    double* o = (double*)j->out;
    for (int64_t i = j->begin; i < j->end; ++i)
      o[i] = (double)(draw_at(j->key, j->first + (uint64_t)i) >> 11) * kInv53;
  }
  return NULL;
}

static void run_parallel(job_t base, int64_t n, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < ((int64_t)1 << 16)) nthreads = 1;
  pthread_t th[256];
  int live[256];
  job_t jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = base;
    jobs[t].begin = n * t / nthreads;
    jobs[t].end = n * (t + 1) / nthreads;
    live[t] = (t + 1 < nthreads) && pthread_create(&th[t], NULL, run_job, &jobs[t]) == 0;
    if (!live[t]) run_job(&jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t)
    if (live[t]) pthread_join(th[t], NULL);
}

SYNTH_API uint64_t synth_draw(uint64_t seed, uint64_t tid, uint64_t i) {
  return draw_at(stream_key(seed, tid), i);
}

SYNTH_API double synth_normal(uint64_t seed, uint64_t tid, uint64_t i) {
  return normal_at(stream_key(seed, tid), i);
}

SYNTH_API uint16_t synth_bf16_of(double x) { return to_bf16(x); }

/* out[i] = bf16(sigma * normal(seed, tid, first + i)), i in [0, n). */
SYNTH_API void synth_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t tid,
                                 uint64_t first, double sigma, int nthreads) {
  job_t b = {0, out, 0, 0, stream_key(seed, tid), first, sigma, 0};
  run_parallel(b, n, nthreads);
}

/* out[i] = draw(seed, tid, first + i) % modulus. */
SYNTH_API void synth_ids(int32_t* out, int64_t n, uint64_t seed, uint64_t tid, uint64_t first,
                         int64_t modulus, int nthreads) {
  job_t b = {1, out, 0, 0, stream_key(seed, tid), first, 0.0, modulus};
  run_parallel(b, n, nthreads);
}

/* out[i] = uniform [0,1) from draw(seed, tid, first + i). */
SYNTH_API void synth_uniform(double* out, int64_t n, uint64_t seed, uint64_t tid, uint64_t first,
                             int nthreads) {
  job_t b = {2, out, 0, 0, stream_key(seed, tid), first, 0.0, 0};
  run_parallel(b, n, nthreads);
}

/* out[i] = uniform [0,1) from draw(seed, tid, idx[i]) (arbitrary indices). */
SYNTH_API void synth_uniform_at(double* out, const uint64_t* idx, int64_t n, uint64_t seed,
                                uint64_t tid) {
  const uint64_t key = stream_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) out[i] = (double)(draw_at(key, idx[i]) >> 11) * kInv53;
}

/* out[i] = draw(seed, tid, idx[i]) % modulus (arbitrary indices). */
SYNTH_API void synth_ids_at(int32_t* out, const uint64_t* idx, int64_t n, uint64_t seed,
                            uint64_t tid, int64_t modulus) {
  const uint64_t key = stream_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(draw_at(key, idx[i]) % (uint64_t)modulus);
}
