/*
 * Seeded synthetic input generator shared by the oracle side and the CUDA side.
 *
 * It draws the random numbers that the workloads are made of and nothing else:
 * no reduction, normalisation, rounding to a storage format, quantisation,
 * GEMM or argmax lives here.  The Python wrapper (synth/__init__.py) turns the
 * fp32 draws into BF16 / FP8 storage with torch library casts.
 *
 * Generator definition (counter-based, so any element can be drawn alone):
 *   mix(z)   = splitmix64 output function applied to state z:
 *              z += 0x9E3779B97F4A7C15;
 *              z  = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *              z  = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *              return z ^ (z >> 31);
 *   key      = mix(seed * 0xD1B54A32D192ED03 + stream)
 *   bits(j)  = mix(key + j)
 *   element i of a normal stream uses bits(2i) and bits(2i+1):
 *     u1 = ((bits(2i)   >> 11) + 1) * 2^-53      in (0, 1]
 *     u2 =  (bits(2i+1) >> 11)      * 2^-53      in [0, 1)
 *     n  = sqrt(-2 ln u1) * cos(2 pi u2)          (Box-Muller, cosine branch)
 *     x  = (float)(mean + std * n)                (double arithmetic)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

static uint64_t mix(uint64_t z) {
  z += 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix(seed * 0xD1B54A32D192ED03ULL + stream);
}

uint64_t synth_bits(uint64_t seed, uint64_t stream, uint64_t j) {
  return mix(stream_key(seed, stream) + j);
}

static double normal_at(uint64_t key, uint64_t i) {
  const double two_m53 = 1.0 / 9007199254740992.0;
  double u1 = (double)((mix(key + 2 * i) >> 11) + 1) * two_m53;
  double u2 = (double)(mix(key + 2 * i + 1) >> 11) * two_m53;
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

typedef struct {
  uint64_t key, start, count;
  double mean, std;
  float *out;
  /* optional per-column multiplier: element i gets mult[i % ncols] */
  const float *colmult;
  uint64_t ncols;
} job_t;

static void *run_job(void *p) {
  job_t *j = (job_t *)p;
  for (uint64_t e = 0; e < j->count; ++e) {
    uint64_t i = j->start + e;
    double x = j->std * normal_at(j->key, i);
    if (j->colmult) x *= (double)j->colmult[i % j->ncols];
    j->out[e] = (float)(j->mean + x);
  }
  return NULL;
}

/* Fill out[0..count) with elements start..start+count-1 of the normal stream
 * (seed, stream) scaled to N(mean, std^2); when colmult is non-NULL the draw of
 * element i (before the mean is added) is multiplied by colmult[i % ncols].
 * Work is split over nthreads POSIX threads; the result does not depend on it. */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count,
                      double mean, double std, const float *colmult, uint64_t ncols,
                      float *out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (count < (1u << 16)) nthreads = 1;
  uint64_t key = stream_key(seed, stream);
  job_t jobs[256];
  pthread_t th[256];
  int started[256] = {0};
  uint64_t per = (count + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
  int launched = 0;
  for (int t = 0; t < nthreads; ++t) {
    uint64_t b = (uint64_t)t * per;
    if (b >= count) break;
    uint64_t n = count - b < per ? count - b : per;
    jobs[t] = (job_t){key, start + b, n, mean, std, out + b, colmult, ncols};
    launched = t + 1;
    if (nthreads == 1 || pthread_create(&th[t], NULL, run_job, &jobs[t]) != 0)
      run_job(&jobs[t]);
    else
      started[t] = 1;
  }
  for (int t = 0; t < launched; ++t)
    if (started[t]) pthread_join(th[t], NULL);
}

/* First n entries of a seeded Fisher-Yates shuffle of 0..len-1 (partial
 * shuffle; position j swaps with j + bits(j) mod (len - j)). */
void synth_choose(uint64_t seed, uint64_t stream, int64_t len, int64_t n, int64_t *out) {
  int64_t *perm = (int64_t *)malloc(sizeof(int64_t) * (size_t)(len > 0 ? len : 1));
  if (!perm) return;
  for (int64_t i = 0; i < len; ++i) perm[i] = i;
  uint64_t key = stream_key(seed, stream);
  for (int64_t j = 0; j < n && j < len; ++j) {
    int64_t r = j + (int64_t)(mix(key + (uint64_t)j) % (uint64_t)(len - j));
    int64_t tmp = perm[j];
    perm[j] = perm[r];
    perm[r] = tmp;
    out[j] = perm[j];
  }
  free(perm);
}
