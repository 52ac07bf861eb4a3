/*
 * Seeded synthetic inputs for the FP4 weight-only linear layer.
 *
 * This module only draws numbers: it holds none of the layer's arithmetic
 * (no FP4/FP8 decoding, no quantisation, no matrix product).  Both the CPU
 * oracle (tests) and the GPU path (tests, benchmarks) take their inputs from
 * here, so the two sides always see the same bf16 tensors.
 *
 * Generator (counter based, so any element or row can be regenerated alone):
 *   base      = mix64(seed * GAMMA + tensor_id)
 *   x_n       = mix64(base + n * GAMMA)            (SplitMix64 output n >= 1)
 *   pair j    : u1 = ((x_{2j+1} >> 11) + 1) * 2^-53   in (0, 1]
 *               u2 =  (x_{2j+2} >> 11)      * 2^-53   in [0, 1)
 *               r  = sqrt(-2 ln u1)
 *               element 2j   = sigma * r * cos(2 pi u2)
 *               element 2j+1 = sigma * r * sin(2 pi u2)      (Box-Muller)
 *   the fp64 value is rounded to fp32 (round to nearest) and then to bf16
 *   (round to nearest, ties to even).
 * mix64 is the SplitMix64 finaliser (Steele, Lea, Flood 2014), GAMMA its
 * golden-ratio increment 0x9E3779B97F4A7C15.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

static double element(uint64_t base, double sigma, int64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t j = (uint64_t)i >> 1;
  uint64_t x1 = mix64(base + (2 * j + 1) * GAMMA);
  uint64_t x2 = mix64(base + (2 * j + 2) * GAMMA);
  double u1 = (double)((x1 >> 11) + 1) * 0x1.0p-53;
  double u2 = (double)(x2 >> 11) * 0x1.0p-53;
  double r = sqrt(-2.0 * log(u1));
  double z = (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
  return sigma * z;
}

typedef struct {
  uint64_t base;
  double sigma;
  const int64_t* starts; /* element index of each run */
  int64_t run_len;       /* elements per run */
  int64_t nruns;
  uint16_t* out;
  int tid, nthreads;
} job_t;

static void* worker(void* p) {
  job_t* jb = (job_t*)p;
  for (int64_t r = jb->tid; r < jb->nruns; r += jb->nthreads) {
    int64_t s = jb->starts ? jb->starts[r] : r * jb->run_len;
    uint16_t* o = jb->out + r * jb->run_len;
    for (int64_t e = 0; e < jb->run_len; ++e)
      o[e] = f32_to_bf16((float)element(jb->base, jb->sigma, s + e));
  }
  return 0;
}

static void run(uint64_t seed, uint64_t tensor_id, double sigma, const int64_t* starts,
                int64_t run_len, int64_t nruns, uint16_t* out, int threads) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t th[256];
  job_t jobs[256];
  uint64_t base = mix64(seed * GAMMA + tensor_id);
  for (int t = 0; t < threads; ++t) {
    jobs[t] = (job_t){base, sigma, starts, run_len, nruns, out, t, threads};
    pthread_create(&th[t], 0, worker, &jobs[t]);
  }
  for (int t = 0; t < threads; ++t) pthread_join(th[t], 0);
}

/* out[r * K + k] = element (r * K + k) of the stream, for r < rows. */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, double sigma, int64_t rows,
                       int64_t K, uint16_t* out, int threads) {
  run(seed, tensor_id, sigma, 0, K, rows, out, threads);
}

/* out[i * K + k] = element (row_idx[i] * K + k): selected rows of a [*, K] tensor. */
void synth_normal_bf16_rows(uint64_t seed, uint64_t tensor_id, double sigma, int64_t K,
                            const int64_t* row_idx, int64_t nrows, uint16_t* out, int threads) {
  int64_t starts_local[4096];
  for (int64_t b = 0; b < nrows; b += 4096) {
    int64_t n = nrows - b < 4096 ? nrows - b : 4096;
    for (int64_t i = 0; i < n; ++i) starts_local[i] = row_idx[b + i] * K;
    run(seed, tensor_id, sigma, starts_local, K, n, out + b * K, threads);
  }
}
