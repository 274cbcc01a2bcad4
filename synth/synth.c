/*
 * Seeded synthetic inputs for the layer-major int8 prefill model.
 *
 * This module only draws data. It holds none of the prefill arithmetic:
 * both the CPU oracle and the CUDA library receive what it produces as
 * plain host arrays.
 *
 * Random numbers: every value is a pure function of (seed, stream, index)
 * through SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), so any thread can draw any slice and
 * every process gets identical bytes. Gaussians come from the Box-Muller
 * transform (Box and Muller, 1958) applied to two uniforms in (0, 1].
 *
 * Weight recipe (the model configs: "int8 symmetric per-output-row with
 * f32 row scales, drawn from N(0, 0.02) then quantised"): for one output
 * row w[0..cols) drawn from N(0, std), scale = max|w| / 127 and
 * code = round-half-away-from-zero(w / scale), all in double, then the
 * scale is stored as f32. This is data preparation of the synthetic
 * checkpoint, not the activation quantiser of the prefill path.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYNTH_TWO_PI 6.283185307179586476925286766559

static inline uint64_t sm64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

/* One 64-bit draw for (seed, stream, index). */
static inline uint64_t draw64(uint64_t seed, uint64_t stream, uint64_t idx) {
  uint64_t key = sm64(seed ^ sm64(stream + 0x632BE59BD9B4E019ull));
  return sm64(key + idx * 0xD1B54A32D192ED03ull);
}

/* Uniform in (0, 1] with 53 random bits. */
static inline double unif(uint64_t r) { return ((double)(r >> 11) + 1.0) * (1.0 / 9007199254740992.0); }

/* Standard normal number idx of a stream (pairs share one Box-Muller draw). */
static inline double normal_at(uint64_t seed, uint64_t stream, uint64_t idx) {
  uint64_t pair = idx >> 1;
  double u1 = unif(draw64(seed, stream, 2 * pair));
  double u2 = unif(draw64(seed, stream, 2 * pair + 1));
  double rad = sqrt(-2.0 * log(u1));
  return (idx & 1) ? rad * sin(SYNTH_TWO_PI * u2) : rad * cos(SYNTH_TWO_PI * u2);
}

typedef struct {
  uint64_t seed, stream;
  int64_t begin, end; /* rows (int8 matrices) or elements (f32 arrays) */
  int64_t cols;
  double mean, std;
  float* f32_out;
  int8_t* q_out;
  float* scale_out;
} job_t;

static void* f32_worker(void* p) {
  job_t* j = (job_t*)p;
  for (int64_t i = j->begin; i < j->end; ++i)
    j->f32_out[i] = (float)(j->mean + j->std * normal_at(j->seed, j->stream, (uint64_t)i));
  return NULL;
}

static void* q8_worker(void* p) {
  job_t* j = (job_t*)p;
  double* row = (double*)malloc(sizeof(double) * (size_t)j->cols);
  for (int64_t r = j->begin; r < j->end; ++r) {
    double amax = 0.0;
    for (int64_t c = 0; c < j->cols; ++c) {
      double v = j->std * normal_at(j->seed, j->stream, (uint64_t)(r * j->cols + c));
      row[c] = v;
      double a = fabs(v);
      if (a > amax) amax = a;
    }
    int8_t* q = j->q_out + r * j->cols;
    if (amax == 0.0) {
      memset(q, 0, (size_t)j->cols);
      j->scale_out[r] = 0.0f;
      continue;
    }
    double s = amax / 127.0;
    for (int64_t c = 0; c < j->cols; ++c) {
      double t = round(row[c] / s); /* C round(): halves away from zero */
      if (t > 127.0) t = 127.0;
      if (t < -127.0) t = -127.0;
      q[c] = (int8_t)t;
    }
    j->scale_out[r] = (float)s;
  }
  free(row);
  return NULL;
}

static void run_jobs(job_t* base, int64_t total, int n_threads, void* (*fn)(void*)) {
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if ((int64_t)n_threads > total) n_threads = (int)(total > 0 ? total : 1);
  pthread_t th[256];
  job_t jobs[256];
  int64_t per = (total + n_threads - 1) / n_threads;
  int started = 0;
  for (int t = 0; t < n_threads; ++t) {
    jobs[t] = *base;
    jobs[t].begin = (int64_t)t * per;
    jobs[t].end = jobs[t].begin + per < total ? jobs[t].begin + per : total;
    if (jobs[t].begin >= jobs[t].end) break;
    if (pthread_create(&th[t], NULL, fn, &jobs[t]) != 0) {
      fn(&jobs[t]); /* no thread available: do the slice here */
      th[t] = (pthread_t)0;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

/* out[i] = mean + std * N(0,1)[seed, stream, i] for i in [0, n). */
void synth_normal_f32(uint64_t seed, uint64_t stream, float* out, int64_t n, double mean, double std,
                      int n_threads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.seed = seed; j.stream = stream; j.mean = mean; j.std = std; j.f32_out = out;
  run_jobs(&j, n, n_threads, f32_worker);
}

/* rows x cols int8 matrix drawn from N(0, std) and quantised per row (see header). */
void synth_int8_rows(uint64_t seed, uint64_t stream, int64_t rows, int64_t cols, double std, int8_t* q,
                     float* scale, int n_threads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.seed = seed; j.stream = stream; j.cols = cols; j.std = std; j.q_out = q; j.scale_out = scale;
  run_jobs(&j, rows, n_threads, q8_worker);
}

/* Token ids uniform in [0, vocab): high 64 bits of draw * vocab (Lemire's multiply-shift). */
void synth_tokens(uint64_t seed, uint64_t stream, int32_t* out, int64_t n, int32_t vocab) {
  for (int64_t i = 0; i < n; ++i) {
    unsigned __int128 m = (unsigned __int128)draw64(seed, stream, (uint64_t)i) * (uint64_t)vocab;
    out[i] = (int32_t)(m >> 64);
  }
}

/* Uniform f32 in [lo, hi) (used for kernel-level test inputs). */
void synth_uniform_f32(uint64_t seed, uint64_t stream, float* out, int64_t n, double lo, double hi) {
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(lo + (hi - lo) * (unif(draw64(seed, stream, (uint64_t)i)) - 0x1p-53));
}

/* Uniform int8 in [lo, hi] (used for kernel-level test inputs). */
void synth_uniform_i8(uint64_t seed, uint64_t stream, int8_t* out, int64_t n, int lo, int hi) {
  uint64_t span = (uint64_t)(hi - lo + 1);
  for (int64_t i = 0; i < n; ++i) {
    unsigned __int128 m = (unsigned __int128)draw64(seed, stream, (uint64_t)i) * span;
    out[i] = (int8_t)(lo + (int)(m >> 64));
  }
}
