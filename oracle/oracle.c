/*
 * ORACLE -- test infrastructure only.
 *
 * A plain, slow, obviously correct CPU implementation of the FP4 weight-only
 * (W4A16) linear layer: NVFP4 and MXFP4 weights against bf16 activations; and of
 * its W4A4 arm, where the activations are quantised to the same block format
 * (orc_quantize_act, orc_gemm_w4a4 at the end of the file).
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library; the product path never does.  It shares no code with the
 * CUDA path.
 *
 * Sources (vllm.cpp pull-request pages):
 *  - "keep the ModelOpt NVFP4 lm_head packed" (PR #263), section "Why this row
 *    matters": an NVFP4 weight is U8 codes, two per byte, plus one FP8 scale
 *    per 16 weights and an FP32 second (global) scale; its footprint is
 *    K*N/2 + K*N/16 bytes ("Round-2 findings resolved", item 4).
 *  - "re-verify 27B NVFP4 on the nvidia ModelOpt checkpoint" (PR #178),
 *    section "Layer 3 -- ModelOpt NVFP4 naming": weight_scale_2 is a direct
 *    multiplier; "W4A16 is the default for ModelOpt": activations stay 16-bit.
 *  - "native MXFP4 keep-quant + Qwen e2e" (PR #38), commit "W2": MXFP4 is
 *    E2M1 codes with one E8M0 (kFE8M0fnu) scale per 32 weights, stored U8
 *    [N, K/32], and no global scale; commit "W3 device unit gate": the check
 *    is the GEMM against a CPU dequantisation to f32 followed by an f32 matmul.
 *  - Bit layouts (the pages only name kFE4M3fn / kFE8M0fnu / E2M1): OCP
 *    Microscaling Formats v1.0 (E2M1, E8M0) and OCP 8-bit Floating Point
 *    (E4M3, "fn": no infinities, S.1111.111 is NaN).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - nibble order: the low nibble of byte k/2 holds the even k;
 *  - layout: codes row-major [N][K/2], scales row-major [N][K/g], K fastest;
 *  - dequantised weight: NVFP4 w = fl32(fl32(c*s) * G) (c*s is exact);
 *    MXFP4 w = c * 2^(e-127) (exact);
 *  - GEMM: y[m][n] = sum_k fp32(A[m][k]) * w[n][k], fp32, increasing k,
 *    products and sums rounded separately (no fused multiply-add); the bf16
 *    output is y rounded to nearest even;
 *  - synthetic quantiser: NVFP4 G = fl32(amax / (6*448)), group scale
 *    s = E4M3_RNE_sat(amax_g / (6 G)), codes = E2M1_RNE_sat(w / (s G));
 *    MXFP4 e = smallest integer with 2^e >= amax_g / 6 (clamped to
 *    [-127, 127]), codes = E2M1_RNE_sat(w / 2^e); quotients in fp64; ties to
 *    even; a magnitude that rounds to 0 gives code 0 (+0); a group whose
 *    scale decodes to 0 gets all-zero codes; an all-zero tensor gets G = 1;
 *  - W4A4 activation quantiser: the same group rules with the activation global
 *    alpha in place of G, decisions in fp32 (see orc_quantize_act).
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_NVFP4 = 0, ORC_MXFP4 = 1 };

/* ---------------------------------------------------------------- formats */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent 0 is subnormal: 0.5 * m.  Otherwise 2^(e-1) * (1 + m/2). */
double orc_e2m1_value(unsigned code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

/* E4M3 (fn): sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.
 * Exponent 0 is subnormal: (F/8) * 2^-6.  S.1111.111 is NaN; no infinities. */
double orc_e4m3_value(unsigned byte) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 15, f = byte & 7;
  if (e == 15 && f == 7) return NAN;
  double v = (e == 0) ? ldexp(f / 8.0, -6) : ldexp(1.0 + f / 8.0, e - 7);
  return s ? -v : v;
}

/* E8M0: 2^(byte - 127); 0xFF is NaN. */
double orc_e8m0_value(unsigned byte) {
  if (byte == 0xFF) return NAN;
  return ldexp(1.0, (int)byte - 127);
}

static double bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static float bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* fp32 -> bf16, round to nearest, ties to the even bf16 pattern: the two
 * neighbouring bf16 values are compared by distance in fp64. */
uint16_t orc_f32_to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if (isnan(x)) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t lo = u & 0xFFFF0000u;
  if (lo == u) return (uint16_t)(u >> 16);
  uint32_t hi = lo + 0x10000u; /* next bf16 away from zero */
  double dlo = fabs((double)x - (double)bits_f32(lo));
  double vhi = ((hi & 0x7FFFFFFFu) == 0x7F800000u)
                   ? copysign(ldexp(1.0, 128), (double)x) /* rounds as if 2^128 existed */
                   : (double)bits_f32(hi);
  double dhi = fabs(vhi - (double)x);
  if (dlo < dhi) return (uint16_t)(lo >> 16);
  if (dhi < dlo) return (uint16_t)(hi >> 16);
  return ((lo >> 16) & 1u) ? (uint16_t)(hi >> 16) : (uint16_t)(lo >> 16);
}

/* Nearest E2M1 magnitude code (0..7) to a >= 0; ties go to the even code;
 * values beyond 6 saturate to 6. */
static int e2m1_nearest_mag(double a) {
  int best = 0;
  double bd = fabs(a - orc_e2m1_value(0));
  for (int c = 1; c < 8; ++c) {
    double d = fabs(a - orc_e2m1_value((unsigned)c));
    if (d < bd || (d == bd && (c & 1) == 0)) {
      best = c;
      bd = d;
    }
  }
  return best;
}

unsigned orc_e2m1_from_real(double q) {
  int mag = e2m1_nearest_mag(fabs(q));
  if (mag == 0) return 0; /* a magnitude that rounds to zero is +0 */
  return (q < 0 ? 8u : 0u) | (unsigned)mag;
}

/* Nearest non-negative finite E4M3 byte (0x00..0x7E) to x >= 0; ties go to
 * the even byte; x at or above 448 saturates to 0x7E (never NaN). */
unsigned orc_e4m3_from_real(double x) {
  if (!(x < orc_e4m3_value(0x7E))) return 0x7E;
  int lo = 0, hi = 0x7E; /* value(lo) <= x < value(hi), bytes increase with value */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (orc_e4m3_value((unsigned)mid) <= x) lo = mid; else hi = mid;
  }
  double dl = x - orc_e4m3_value((unsigned)lo), dh = orc_e4m3_value((unsigned)hi) - x;
  if (dl < dh) return (unsigned)lo;
  if (dh < dl) return (unsigned)hi;
  return (lo & 1) ? (unsigned)hi : (unsigned)lo;
}

/* Smallest integer e with 2^e >= amax / 6, i.e. 6 * 2^e >= amax (compared
 * exactly), clamped to [-127, 127]; amax == 0 gives -127. */
int orc_mx_exponent(double amax) {
  if (amax == 0.0) return -127;
  int e = (int)ceil(log2(amax / 6.0));
  while (ldexp(6.0, e - 1) >= amax) --e;
  while (ldexp(6.0, e) < amax) ++e;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* ------------------------------------------------------------- threading */

typedef void (*range_fn)(void* ctx, int64_t begin, int64_t end);
typedef struct {
  range_fn fn;
  void* ctx;
  int64_t n;
  int tid, nthreads;
} pjob_t;

static void* pworker(void* p) {
  pjob_t* j = (pjob_t*)p;
  int64_t b = j->n * j->tid / j->nthreads, e = j->n * (j->tid + 1) / j->nthreads;
  if (e > b) j->fn(j->ctx, b, e);
  return 0;
}

static void parallel_for(int64_t n, int threads, range_fn fn, void* ctx) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (threads == 1 || n < 2) {
    fn(ctx, 0, n);
    return;
  }
  pthread_t th[256];
  pjob_t jobs[256];
  for (int t = 0; t < threads; ++t) {
    jobs[t] = (pjob_t){fn, ctx, n, t, threads};
    pthread_create(&th[t], 0, pworker, &jobs[t]);
  }
  for (int t = 0; t < threads; ++t) pthread_join(th[t], 0);
}

/* ------------------------------------------------------------- quantiser */

typedef struct {
  const uint16_t* W;
  int64_t K;
  int fmt;
  double G;
  uint8_t* codes;
  uint8_t* scales;
} qctx_t;

static void put_code(uint8_t* codes, int64_t K, int64_t n, int64_t k, unsigned c) {
  uint8_t* b = &codes[n * (K / 2) + k / 2];
  if (k % 2 == 0) *b = (uint8_t)((*b & 0xF0u) | c);
  else *b = (uint8_t)((*b & 0x0Fu) | (c << 4));
}

static void quant_rows(void* p, int64_t b, int64_t e) {
  qctx_t* q = (qctx_t*)p;
  const int64_t K = q->K;
  const int g = (q->fmt == ORC_NVFP4) ? 16 : 32;
  for (int64_t n = b; n < e; ++n) {
    for (int64_t grp = 0; grp < K / g; ++grp) {
      const uint16_t* w = q->W + n * K + grp * g;
      double amax_g = 0.0;
      for (int i = 0; i < g; ++i) amax_g = fmax(amax_g, fabs(bf16_value(w[i])));
      double denom;
      if (q->fmt == ORC_NVFP4) {
        unsigned sb = orc_e4m3_from_real(amax_g / (6.0 * q->G));
        q->scales[n * (K / g) + grp] = (uint8_t)sb;
        denom = orc_e4m3_value(sb) * q->G;
      } else {
        int ex = orc_mx_exponent(amax_g);
        q->scales[n * (K / g) + grp] = (uint8_t)(ex + 127);
        denom = ldexp(1.0, ex);
      }
      for (int i = 0; i < g; ++i) {
        unsigned c = (denom == 0.0) ? 0u : orc_e2m1_from_real(bf16_value(w[i]) / denom);
        put_code(q->codes, K, n, grp * g + i, c);
      }
    }
  }
}

typedef struct {
  const uint16_t* W;
  int64_t N, K, chunks;
  double* amax; /* one slot per chunk */
} actx_t;

static void amax_chunks(void* p, int64_t b, int64_t e) {
  actx_t* a = (actx_t*)p;
  for (int64_t c = b; c < e; ++c) {
    int64_t r0 = a->N * c / a->chunks, r1 = a->N * (c + 1) / a->chunks;
    double m = 0.0;
    for (int64_t i = r0 * a->K; i < r1 * a->K; ++i) {
      double v = fabs(bf16_value(a->W[i]));
      if (!(v <= m)) m = v; /* NaN and inf propagate */
    }
    a->amax[c] = m;
  }
}

/* NVFP4 quantiser for synthetic weights.  W: bf16 bits [N][K].  Writes codes
 * [N][K/2], E4M3 scales [N][K/16] and the fp32 global.  Returns 0, or -1 for
 * bad sizes or non-finite input. */
int orc_quantize_nvfp4(const uint16_t* W, int64_t N, int64_t K, uint8_t* codes,
                       uint8_t* scales, float* global_out, int threads) {
  if (N <= 0 || K <= 0 || K % 16) return -1;
  double pam[1024];
  actx_t a = {W, N, K, N < 1024 ? N : 1024, pam};
  parallel_for(a.chunks, threads, amax_chunks, &a);
  double amax = 0.0;
  for (int64_t c = 0; c < a.chunks; ++c)
    if (!(pam[c] <= amax)) amax = pam[c];
  if (!isfinite(amax)) return -1;
  float G = amax > 0.0 ? (float)(amax / (6.0 * 448.0)) : 1.0f;
  qctx_t q = {W, K, ORC_NVFP4, (double)G, codes, scales};
  memset(codes, 0, (size_t)(N * (K / 2)));
  parallel_for(N, threads, quant_rows, &q);
  *global_out = G;
  return 0;
}

/* MXFP4 quantiser for synthetic weights (no global scale). */
int orc_quantize_mxfp4(const uint16_t* W, int64_t N, int64_t K, uint8_t* codes,
                       uint8_t* scales, int threads) {
  if (N <= 0 || K <= 0 || K % 32) return -1;
  for (int64_t i = 0; i < N * K; ++i)
    if (!isfinite(bf16_value(W[i]))) return -1;
  qctx_t q = {W, K, ORC_MXFP4, 1.0, codes, scales};
  memset(codes, 0, (size_t)(N * (K / 2)));
  parallel_for(N, threads, quant_rows, &q);
  return 0;
}

/* ------------------------------------------------------ dequant and GEMM */

static unsigned get_code(const uint8_t* codes, int64_t K, int64_t n, int64_t k) {
  uint8_t b = codes[n * (K / 2) + k / 2];
  return (k % 2 == 0) ? (b & 0x0Fu) : (b >> 4);
}

/* The weight w[n][k] as the layer uses it, in fp32. */
static float weight_f32(int fmt, const uint8_t* codes, const uint8_t* scales, float G,
                        int64_t K, int64_t n, int64_t k) {
  double c = orc_e2m1_value(get_code(codes, K, n, k));
  if (fmt == ORC_NVFP4) {
    float cs = (float)(c * orc_e4m3_value(scales[n * (K / 16) + k / 16])); /* exact */
    return cs * G;                                                        /* one rounding */
  }
  return (float)(c * orc_e8m0_value(scales[n * (K / 32) + k / 32])); /* exact */
}

typedef struct {
  int fmt;
  const uint8_t* codes;
  const uint8_t* scales;
  float G;
  int64_t K;
  float* out;
} dctx_t;

static void dequant_rows(void* p, int64_t b, int64_t e) {
  dctx_t* d = (dctx_t*)p;
  for (int64_t n = b; n < e; ++n)
    for (int64_t k = 0; k < d->K; ++k)
      d->out[n * d->K + k] = weight_f32(d->fmt, d->codes, d->scales, d->G, d->K, n, k);
}

/* out[n][k] = w[n][k] (fp32). */
int orc_dequant(int fmt, const uint8_t* codes, const uint8_t* scales, float G, int64_t N,
                int64_t K, float* out, int threads) {
  if (N <= 0 || K <= 0 || K % (fmt == ORC_NVFP4 ? 16 : 32)) return -1;
  dctx_t d = {fmt, codes, scales, G, K, out};
  parallel_for(N, threads, dequant_rows, &d);
  return 0;
}

typedef struct {
  int fmt;
  const float* A; /* [M][K] fp32 copies of the bf16 activations */
  int64_t M, K, N;
  const uint8_t* codes;
  const uint8_t* scales;
  float G;
  const int64_t* cols; /* NULL: all n in order */
  int64_t ncols;
  float* y;            /* [M][ncols] */
  double* y64;         /* optional [M][ncols] fp64 sums */
  uint16_t* ybf;       /* optional [M][ncols] bf16 */
} gctx_t;

static void gemm_cols(void* p, int64_t b, int64_t e) {
  gctx_t* g = (gctx_t*)p;
  const int64_t K = g->K;
  float* w = (float*)malloc((size_t)K * sizeof(float));
  for (int64_t j = b; j < e; ++j) {
    int64_t n = g->cols ? g->cols[j] : j;
    for (int64_t k = 0; k < K; ++k) w[k] = weight_f32(g->fmt, g->codes, g->scales, g->G, K, n, k);
    for (int64_t m = 0; m < g->M; ++m) {
      const float* a = g->A + m * K;
      float acc = 0.0f;
      double acc64 = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        float prod = a[k] * w[k];
        acc = acc + prod;
        acc64 += (double)a[k] * (double)w[k];
      }
      g->y[m * g->ncols + j] = acc;
      if (g->y64) g->y64[m * g->ncols + j] = acc64;
      if (g->ybf) g->ybf[m * g->ncols + j] = orc_f32_to_bf16(acc);
    }
  }
  free(w);
}

int orc_gemm_f32a(int fmt, const float* Af, int64_t M, int64_t K, const uint8_t* codes,
                  const uint8_t* scales, float G, int64_t N, const int64_t* cols, int64_t ncols,
                  float* y, double* y64, uint16_t* ybf, int threads);

/* y[m][j] = sum_k fp32(A[m][k]) * w[cols[j]][k] (fp32, increasing k); A is bf16
 * bits [M][K] row-major.  cols == NULL computes all N columns.  y64 (optional)
 * receives the same sum accumulated in fp64; ybf (optional) the bf16 output. */
int orc_gemm(int fmt, const uint16_t* A, int64_t M, int64_t K, const uint8_t* codes,
             const uint8_t* scales, float G, int64_t N, const int64_t* cols, int64_t ncols,
             float* y, double* y64, uint16_t* ybf, int threads) {
  if (M < 0 || K <= 0) return -1;
  float* Af = (float*)malloc((size_t)(M * K + 1) * sizeof(float));
  if (!Af) return -1;
  for (int64_t i = 0; i < M * K; ++i) Af[i] = (float)bf16_value(A[i]);
  const int rc = orc_gemm_f32a(fmt, Af, M, K, codes, scales, G, N, cols, ncols, y, y64, ybf,
                               threads);
  free(Af);
  return rc;
}

/* The same GEMM with the activations already in fp32 ([M][K], row-major): the W4A4 layer,
 * whose activations are the dequantised FP4 values fl32(fl32(c s) G_a) (or c 2^(e-127)). */
int orc_gemm_f32a(int fmt, const float* Af, int64_t M, int64_t K, const uint8_t* codes,
                  const uint8_t* scales, float G, int64_t N, const int64_t* cols, int64_t ncols,
                  float* y, double* y64, uint16_t* ybf, int threads) {
  if (M < 0 || N <= 0 || K <= 0 || K % (fmt == ORC_NVFP4 ? 16 : 32)) return -1;
  if (!cols) ncols = N;
  for (int64_t j = 0; cols && j < ncols; ++j)
    if (cols[j] < 0 || cols[j] >= N) return -1;
  gctx_t g = {fmt, Af, M, K, N, codes, scales, G, cols, ncols, y, y64, ybf};
  parallel_for(ncols, threads, gemm_cols, &g);
  return 0;
}

/* ------------------------------------------------------------ greedy head */
/* Greedy token choice over each row of bf16 outputs ybf [M][N]: the index of the largest
 * value, and among equal values the lowest index.  Source: "re-verify 27B NVFP4 on the
 * nvidia ModelOpt checkpoint" (PR #178), section "Correctness -- resolved, not fixed": the
 * greedy argmax breaks a tie by the lowest index (on the true global index); section
 * "Speed -- warp-shuffle MoE router top-k": under that total order the argmax gives the
 * same (value, index) in any reduction order.  Values compare as numbers, so -0 equals +0;
 * a NaN counts as larger than every number and the first NaN wins (a NaN-propagating
 * argmax).  val (optional) receives the chosen bf16 value. */
static int greedy_better(double a, double b) {
  if (isnan(b)) return 0;
  if (isnan(a)) return 1;
  return a > b;
}

int orc_greedy(const uint16_t* ybf, int64_t M, int64_t N, int32_t* idx, uint16_t* val) {
  if (M < 0 || N <= 0 || N > 2147483647LL) return -1;
  for (int64_t m = 0; m < M; ++m) {
    const uint16_t* row = ybf + m * N;
    int64_t best = 0;
    for (int64_t n = 1; n < N; ++n)
      if (greedy_better(bf16_value(row[n]), bf16_value(row[best]))) best = n;
    idx[m] = (int32_t)best;
    if (val) val[m] = row[best];
  }
  return 0;
}

/* ---------------------------------------------------- SiLU-gated MLP input */
/* fp64 -> bf16, one rounding to nearest (ties to even): 8 significant bits for normal
 * values, multiples of 2^-133 below 2^-126, infinity past the largest bf16. */
static uint16_t f64_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  const double a = fabs(x);
  int e = 0;
  const double mnt = frexp(a, &e);  /* a = mnt * 2^e, mnt in [0.5, 1) */
  double q;
  if (a == 0.0) q = 0.0;
  else if (e - 1 >= -126) q = ldexp(rint(ldexp(mnt, 8)), e - 8);
  else q = ldexp(rint(ldexp(a, 133)), -133);
  const float f = (q >= 0x1p128) ? INFINITY : (float)q; /* exact: q fits bf16 */
  return orc_f32_to_bf16(signbit(x) ? -f : f);
}

/* The input of the down projection from a fused gate_up output: for gate and up sums
 * g = y[m][i] and u = y[m][I + i] (fp32, as the GEMM sums them),
 *   out[m][i] = bf16_RNE( silu(g) * u ),  silu(x) = x / (1 + e^-x),
 * evaluated in fp64 from the fp32 sums.  Source: "MXFP4 decode-graph + gate_up FUSION
 * default-ON" (PR #54), "Step 2": gate and up are one GEMM of N = 2I whose halves feed the
 * SiLU-and-multiply step before down; "Attribution": that glue between the GEMMs is a
 * measured cost of the decode step. */
int orc_silu_mul(const float* y, int64_t M, int64_t I, uint16_t* out) {
  if (M < 0 || I <= 0) return -1;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t i = 0; i < I; ++i) {
      const double g = (double)y[m * 2 * I + i], u = (double)y[m * 2 * I + I + i];
      const double s = g / (1.0 + exp(-g));
      out[m * I + i] = f64_to_bf16(s * u);
    }
  return 0;
}

/* ------------------------------------------------------ W4A4 activations */
/* The W4A4 arm quantises the activations too, with the same block formats as the weights:
 * NVFP4 with the per-tensor activation global alpha (the checkpoint's "input_scale", which
 * sets the GEMM's alpha and makes the layer true W4A4), MXFP4 with no global.  "re-verify 27B
 * NVFP4 on the nvidia ModelOpt checkpoint" (PR #178), section "W4A16 is the default for
 * ModelOpt"; "native MXFP4 keep-quant + Qwen e2e" (PR #38), commit "W0" (input_activations
 * set = true W4A4).  The pages fix no precision for this quantiser; here every rounding
 * decision is taken in fp32 (IEEE, round to nearest even), the precision of the GPU kernels:
 *   NVFP4: s = E4M3_RNE_sat(fl32(amax_g / fl32(6 alpha))), d = fl32(val(s) alpha),
 *          c = E2M1_RNE_sat(fl32(x / d))  (c = 0 for the whole group when s = 0);
 *          dequantised a = fl32(fl32(val(c) val(s)) alpha).
 *   MXFP4: e = min{e : 6 2^e >= amax_g} clamped to [-127, 127] (exact),
 *          c = E2M1_RNE_sat(fl32(x fl32(2^-e))); dequantised a = fl32(val(c) 2^e).
 * A: bf16 bits [M][K]; codes [M][K/2] (low nibble first), scales [M][K/g]; Aq (optional)
 * [M][K] fp32 dequantised activations.  Returns -1 for bad sizes, a non-finite input, or
 * (NVFP4) an alpha that is not a positive normal float; MXFP4 requires alpha == 1. */
typedef struct {
  const uint16_t* A;
  int64_t K;
  int fmt;
  float alpha;
  uint8_t* codes;
  uint8_t* scales;
  float* Aq;
} aqctx_t;

static void act_quant_rows(void* p, int64_t b, int64_t e) {
  aqctx_t* q = (aqctx_t*)p;
  const int64_t K = q->K;
  const int g = (q->fmt == ORC_NVFP4) ? 16 : 32;
  const float alpha6 = 6.0f * q->alpha;
  for (int64_t m = b; m < e; ++m) {
    for (int64_t grp = 0; grp < K / g; ++grp) {
      const uint16_t* x = q->A + m * K + grp * g;
      float amax = 0.0f;
      for (int i = 0; i < g; ++i) amax = fmaxf(amax, fabsf((float)bf16_value(x[i])));
      float d, step;
      if (q->fmt == ORC_NVFP4) {
        const float qs = amax / alpha6;
        const unsigned sb = orc_e4m3_from_real((double)qs);
        q->scales[m * (K / g) + grp] = (uint8_t)sb;
        step = (float)orc_e4m3_value(sb);
        d = step * q->alpha;
      } else {
        const int ex = orc_mx_exponent((double)amax);
        q->scales[m * (K / g) + grp] = (uint8_t)(ex + 127);
        step = ldexpf(1.0f, ex);
        d = ldexpf(1.0f, -ex); /* multiplier for MXFP4 */
      }
      for (int i = 0; i < g; ++i) {
        const float xv = (float)bf16_value(x[i]);
        unsigned c;
        if (q->fmt == ORC_NVFP4) c = (step == 0.0f) ? 0u : orc_e2m1_from_real((double)(xv / d));
        else c = orc_e2m1_from_real((double)(xv * d));
        put_code(q->codes, K, m, grp * g + i, c);
        if (q->Aq) {
          const float cv = (float)orc_e2m1_value(c);
          q->Aq[m * K + grp * g + i] =
              (q->fmt == ORC_NVFP4) ? (cv * step) * q->alpha : cv * step;
        }
      }
    }
  }
}

int orc_quantize_act(int fmt, const uint16_t* A, int64_t M, int64_t K, float alpha,
                     uint8_t* codes, uint8_t* scales, float* Aq, int threads) {
  if (M <= 0 || K <= 0 || K % (fmt == ORC_NVFP4 ? 16 : 32)) return -1;
  if (fmt == ORC_NVFP4 ? !(isfinite(alpha) && alpha >= FLT_MIN) : alpha != 1.0f) return -1;
  for (int64_t i = 0; i < M * K; ++i)
    if (!isfinite(bf16_value(A[i]))) return -1;
  aqctx_t q = {A, K, fmt, alpha, codes, scales, Aq};
  memset(codes, 0, (size_t)(M * (K / 2)));
  parallel_for(M, threads, act_quant_rows, &q);
  return 0;
}

/* The W4A4 layer: y[m][j] = sum_k a[m][k] w[cols[j]][k] in fp32 (increasing k) with a the
 * dequantised activations of orc_quantize_act and w the dequantised weights, the same
 * accumulation as orc_gemm; y64 and ybf as there. */
int orc_gemm_w4a4(int fmt, const uint16_t* A, int64_t M, int64_t K, float alpha,
                  const uint8_t* codes, const uint8_t* scales, float G, int64_t N,
                  const int64_t* cols, int64_t ncols, float* y, double* y64, uint16_t* ybf,
                  int threads) {
  if (M <= 0 || K <= 0) return -1;
  const int g = (fmt == ORC_NVFP4) ? 16 : 32;
  if (K % g) return -1;
  uint8_t* ac = (uint8_t*)malloc((size_t)(M * (K / 2)));
  uint8_t* as = (uint8_t*)malloc((size_t)(M * (K / g)));
  float* Aq = (float*)malloc((size_t)(M * K) * sizeof(float));
  int rc = -1;
  if (ac && as && Aq && orc_quantize_act(fmt, A, M, K, alpha, ac, as, Aq, threads) == 0)
    rc = orc_gemm_f32a(fmt, Aq, M, K, codes, scales, G, N, cols, ncols, y, y64, ybf, threads);
  free(ac);
  free(as);
  free(Aq);
  return rc;
}
