/*
 * Seeded synthetic inputs for masked attention over a BlockMask.
 *
 * This module holds no part of the attention method: it only turns
 * (seed, tensor id, element index) into numbers, so that the CPU oracle and
 * the CUDA path read byte-identical inputs.
 *
 *  - splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *    generators", OOPSLA 2014; the public-domain reference generator by
 *    Vigna): state += 0x9E3779B97F4A7C15, output = mix(state).
 *    Stream (seed, tid) is the splitmix64 generator whose initial state is
 *    mix(seed + tid * gamma); draw k is its (k+1)-th output, so any element
 *    can be produced independently of the others (counter based).
 *  - Box-Muller transform (Box and Muller, 1958) on pairs of draws
 *    (2p, 2p+1): element 2p takes r*cos(theta), element 2p+1 r*sin(theta).
 *  - bf16 round-to-nearest-even taken directly from the fp64 value.
 *  - Integer draws uniform on [lo, hi] by rejection (no modulo bias), taken
 *    sequentially from the stream; Fisher-Yates shuffle from those draws.
 *
 * Plain C99 + pthreads; no architecture-specific code.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_stream_state(uint64_t seed, uint64_t tid) {
  return sm_mix(seed + tid * SM_GAMMA);
}

/* k-th output (k >= 0) of the splitmix64 generator started at `state`. */
static inline uint64_t sm_draw(uint64_t state, uint64_t k) {
  return sm_mix(state + (k + 1) * SM_GAMMA);
}

uint64_t synth_draw_u64(uint64_t seed, uint64_t tid, uint64_t k) {
  return sm_draw(synth_stream_state(seed, tid), k);
}

/* (x >> 11 + 0.5) * 2^-53: uniform on the open interval (0, 1). */
static inline double sm_unit(uint64_t x) {
  return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double sm_normal(uint64_t state, uint64_t e) {
  uint64_t p = e >> 1;
  double u1 = sm_unit(sm_draw(state, 2 * p));
  double u2 = sm_unit(sm_draw(state, 2 * p + 1));
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  return (e & 1) ? r * sin(th) : r * cos(th);
}

/* Round an fp64 value to the nearest bf16 (ties to even) and return its bits.
 * Rounds the fp64 significand to 8 bits first; the result is then exactly
 * representable in fp32 and bf16, so the narrowing casts below are exact. */
static inline uint16_t sm_bf16_rne(double x) {
  if (x != x) return 0x7FC0;
  uint64_t b;
  memcpy(&b, &x, 8);
  uint64_t lsb = (b >> 45) & 1ULL;
  b += 0x0000100000000000ULL - 1ULL + lsb; /* 2^44 - 1 + lsb */
  b &= ~((1ULL << 45) - 1ULL);
  double y;
  memcpy(&y, &b, 8);
  float f = (float)y; /* exact unless it overflows to inf, which is the bf16 answer too */
  uint32_t fb;
  memcpy(&fb, &f, 4);
  return (uint16_t)(fb >> 16);
}

uint16_t synth_bf16_from_double(double x) { return sm_bf16_rne(x); }

typedef struct {
  uint64_t state, first, count;
  double mean, stddev;
  uint16_t* out_bf16;
  double* out_f64;
} sm_job;

static void* sm_worker(void* arg) {
  sm_job* j = (sm_job*)arg;
  for (uint64_t i = 0; i < j->count; ++i) {
    double v = j->mean + j->stddev * sm_normal(j->state, j->first + i);
    if (j->out_bf16) j->out_bf16[i] = sm_bf16_rne(v);
    if (j->out_f64) j->out_f64[i] = v;
  }
  return NULL;
}

static int sm_threads(uint64_t count) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  if (n < 1) n = 1;
  if (n > 64) n = 64;
  uint64_t per = 1u << 16;
  if (count / per + 1 < (uint64_t)n) n = (long)(count / per + 1);
  return (int)n;
}

static void sm_run(uint64_t seed, uint64_t tid, uint64_t first, uint64_t count,
                   double mean, double stddev, uint16_t* ob, double* od) {
  uint64_t state = synth_stream_state(seed, tid);
  int nt = sm_threads(count);
  sm_job jobs[64];
  pthread_t th[64];
  uint64_t per = (count + (uint64_t)nt - 1) / (uint64_t)nt;
  int launched = 0;
  for (int t = 0; t < nt; ++t) {
    uint64_t a = (uint64_t)t * per;
    if (a >= count) break;
    uint64_t n = count - a < per ? count - a : per;
    jobs[t].state = state;
    jobs[t].first = first + a;
    jobs[t].count = n;
    jobs[t].mean = mean;
    jobs[t].stddev = stddev;
    jobs[t].out_bf16 = ob ? ob + a : NULL;
    jobs[t].out_f64 = od ? od + a : NULL;
    if (nt == 1 || pthread_create(&th[t], NULL, sm_worker, &jobs[t]) != 0) {
      sm_worker(&jobs[t]);
      th[t] = 0;
    }
    launched = t + 1;
  }
  for (int t = 0; t < launched; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

/* Elements [first, first+count) of stream (seed, tid) as N(mean, stddev^2), rounded to bf16. */
void synth_normal_bf16(uint64_t seed, uint64_t tid, uint64_t first, uint64_t count,
                       double mean, double stddev, uint16_t* out) {
  sm_run(seed, tid, first, count, mean, stddev, out, NULL);
}

/* Same stream, unrounded fp64 values (used to check the rounding step). */
void synth_normal_f64(uint64_t seed, uint64_t tid, uint64_t first, uint64_t count,
                      double mean, double stddev, double* out) {
  sm_run(seed, tid, first, count, mean, stddev, NULL, out);
}

/* Sequential integer draws uniform on [lo, hi] (inclusive) from stream (seed, tid),
 * starting at draw *cursor; *cursor is advanced past every draw consumed,
 * rejected ones included. */
void synth_uniform_int(uint64_t seed, uint64_t tid, uint64_t* cursor, int64_t lo, int64_t hi,
                       int64_t count, int64_t* out) {
  uint64_t state = synth_stream_state(seed, tid);
  uint64_t range = (uint64_t)(hi - lo) + 1ULL;
  /* largest multiple of range that fits in 2^64 (range == 0 means all 2^64 values) */
  uint64_t limit = range ? (0ULL - ((0ULL - range) % range)) : 0ULL;
  uint64_t k = *cursor;
  for (int64_t i = 0; i < count; ++i) {
    uint64_t x;
    for (;;) {
      x = sm_draw(state, k++);
      if (range == 0 || limit == 0 || x < limit) break;
    }
    out[i] = range ? lo + (int64_t)(x % range) : (int64_t)x;
  }
  *cursor = k;
}

/* Fisher-Yates: out = a permutation of [0, n) drawn from stream (seed, tid). */
void synth_permutation(uint64_t seed, uint64_t tid, int64_t n, int32_t* out) {
  uint64_t cursor = 0;
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (int64_t i = n - 1; i >= 1; --i) {
    int64_t j;
    synth_uniform_int(seed, tid, &cursor, 0, i, 1, &j);
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}
