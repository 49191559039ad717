/*
 * Seeded synthetic input generators for the MoE routing workloads.
 *
 * Shared by the oracle's tests, the GPU parity tests and the benchmark: this
 * file produces input tensors only and holds none of the routing, indexing or
 * combine arithmetic.
 *
 * Generator (counter based, so any element range can be regenerated on its own):
 *   key(seed, tensor)  = mix64(seed * 0x9E3779B97F4A7C15 + tensor)
 *   bits(key, c)       = mix64(key + (c + 1) * 0x9E3779B97F4A7C15)
 *   uniform(key, c)    = ((bits >> 11) + 0.5) * 2^-53          in (0, 1)
 * where mix64 is the SplitMix64 output function (Steele, Lea, Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014).
 * Standard normals come in Box-Muller pairs: pair j takes u1 = uniform(key, 2j)
 * and u2 = uniform(key, 2j + 1), r = sqrt(-2 ln u1), and element 2j is
 * r cos(2 pi u2), element 2j + 1 is r sin(2 pi u2) (Box and Muller 1958).
 * Every transform is evaluated in double and rounded once to float
 * (round-to-nearest-even); bf16 values are the float rounded to nearest-even.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor) {
  return mix64(seed * GOLDEN + tensor);
}

static inline double uniform01(uint64_t key, uint64_t c) {
  uint64_t b = mix64(key + (c + 1) * GOLDEN);
  return ((double)(b >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Standard normal number i of the stream. */
static inline double normal_at(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t j = i >> 1;
  double u1 = uniform01(key, 2 * j);
  double u2 = uniform01(key, 2 * j + 1);
  double r = sqrt(-2.0 * log(u1));
  return (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

enum { K_NORMAL_F32 = 0, K_SIGMOID_F32 = 1, K_BF16 = 2, K_SOFTMAX_ROWS = 3 };

typedef struct {
  int kind;
  uint64_t key;
  int64_t first; /* first element (or row) index of the stream */
  int64_t begin, end; /* this worker's range, relative to `first` */
  int64_t cols;       /* softmax row length */
  double mean, std;
  void *out;
} job_t;

static void run_range(const job_t *j) {
  if (j->kind == K_NORMAL_F32) {
    float *o = (float *)j->out;
    for (int64_t i = j->begin; i < j->end; ++i)
      o[i] = (float)(j->mean + j->std * normal_at(j->key, (uint64_t)(j->first + i)));
  } else if (j->kind == K_SIGMOID_F32) {
    float *o = (float *)j->out;
    for (int64_t i = j->begin; i < j->end; ++i) {
      double z = normal_at(j->key, (uint64_t)(j->first + i));
      o[i] = (float)(1.0 / (1.0 + exp(-z)));
    }
  } else if (j->kind == K_BF16) {
    uint16_t *o = (uint16_t *)j->out;
    int64_t i = j->begin;
    /* whole Box-Muller pairs share one log/sqrt */
    const double two_pi = 6.283185307179586476925286766559;
    while (i < j->end) {
      uint64_t g = (uint64_t)(j->first + i);
      if ((g & 1) == 0 && i + 1 < j->end) {
        uint64_t p = g >> 1;
        double u1 = uniform01(j->key, 2 * p), u2 = uniform01(j->key, 2 * p + 1);
        double r = sqrt(-2.0 * log(u1));
        o[i] = f32_to_bf16_rne((float)(r * cos(two_pi * u2)));
        o[i + 1] = f32_to_bf16_rne((float)(r * sin(two_pi * u2)));
        i += 2;
      } else {
        o[i] = f32_to_bf16_rne((float)normal_at(j->key, g));
        i += 1;
      }
    }
  } else { /* K_SOFTMAX_ROWS: row-wise softmax of standard-normal logits */
    float *o = (float *)j->out;
    int64_t C = j->cols;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(C > 0 ? C : 1));
    for (int64_t r = j->begin; r < j->end; ++r) {
      uint64_t base = (uint64_t)(j->first + r) * (uint64_t)C;
      double m = -INFINITY, s = 0.0;
      for (int64_t c = 0; c < C; ++c) {
        tmp[c] = normal_at(j->key, base + (uint64_t)c);
        if (tmp[c] > m) m = tmp[c];
      }
      for (int64_t c = 0; c < C; ++c) { tmp[c] = exp(tmp[c] - m); s += tmp[c]; }
      for (int64_t c = 0; c < C; ++c) o[r * C + c] = (float)(tmp[c] / s);
    }
    free(tmp);
  }
}

static void *worker(void *arg) {
  run_range((const job_t *)arg);
  return NULL;
}

static void run_parallel(job_t proto, int64_t n, int nthreads) {
  if (nthreads <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = c > 0 ? (int)c : 1;
  }
  if (nthreads > 256) nthreads = 256;
  int64_t min_per = (proto.kind == K_SOFTMAX_ROWS) ? 64 : 65536;
  if ((int64_t)nthreads * min_per > n) nthreads = (int)((n + min_per - 1) / min_per);
  if (nthreads <= 1) {
    proto.begin = 0;
    proto.end = n;
    run_range(&proto);
    return;
  }
  pthread_t th[256];
  job_t jobs[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  per += per & 1; /* keep Box-Muller pairs inside one worker where possible */
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].begin = (int64_t)t * per;
    jobs[t].end = jobs[t].begin + per < n ? jobs[t].begin + per : n;
    if (jobs[t].begin >= n) break;
    if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) {
      run_range(&jobs[t]);
      jobs[t].kind = -1;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (jobs[t].kind != -1) pthread_join(th[t], NULL);
}

/* out[i] = float(mean + std * z(first + i)), i < n */
void synth_normal_f32(uint64_t seed, uint64_t tensor, double mean, double std, float *out,
                      int64_t first, int64_t n, int nthreads) {
  job_t j = {K_NORMAL_F32, stream_key(seed, tensor), first, 0, 0, 0, mean, std, out};
  run_parallel(j, n, nthreads);
}

/* out[i] = float(1 / (1 + exp(-z(first + i)))) */
void synth_sigmoid_normal_f32(uint64_t seed, uint64_t tensor, float *out, int64_t first, int64_t n,
                              int nthreads) {
  job_t j = {K_SIGMOID_F32, stream_key(seed, tensor), first, 0, 0, 0, 0.0, 1.0, out};
  run_parallel(j, n, nthreads);
}

/* out[r, c] = softmax over c of z((first + r) * cols + c), rows x cols floats */
void synth_softmax_normal_f32(uint64_t seed, uint64_t tensor, float *out, int64_t first_row,
                              int64_t rows, int64_t cols, int nthreads) {
  job_t j = {K_SOFTMAX_ROWS, stream_key(seed, tensor), first_row, 0, 0, cols, 0.0, 1.0, out};
  run_parallel(j, rows, nthreads);
}

/* out[i] = bf16_rne(float(z(first + i))) as raw 16-bit patterns */
void synth_normal_bf16(uint64_t seed, uint64_t tensor, uint16_t *out, int64_t first, int64_t n,
                       int nthreads) {
  job_t j = {K_BF16, stream_key(seed, tensor), first, 0, 0, 0, 0.0, 1.0, out};
  run_parallel(j, n, nthreads);
}
