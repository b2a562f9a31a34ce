/*
 * CPU oracle for the BF16 TN GEMM — TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg call
 * this file.  The product path (the CUDA library) never links or calls it,
 * and it shares no code, header or constant with that library.
 *
 * What it computes is the plain definition of the operation, in FP64:
 *
 *   ref[i][j] = alpha * sum_{k<K} a(i,k) * b(j,k)  +  beta * c(i,j)
 *
 * with a(i,k) = A[i*lda + k], b(j,k) = B[j*ldb + k] (both operands K-major,
 * the "TN" convention of the SM80_16x8x16_F32F16F16F32_TN atom named on the
 * FlashAttention SM80 kernel page, section on the SM80 mainloop), and
 * c(i,j) = C[i*ldc + j] (row-major, N contiguous).  The product-sum is the
 * GEMM work the H100 Nsight Compute page counts as F = 2MNK (section 7,
 * "connecting reuse, capacity and throughput with GEMM"); the "+ beta*C"
 * term is the D <- A*B + C accumulate form the Ampere-to-Hopper page
 * discusses for WGMMA (section "WGMMA", scale_d).
 *
 * bf16 decoding: a bf16 value is the upper 16 bits of an IEEE binary32, so
 * decoding shifts the 16 bits left by 16 and reinterprets them as a float,
 * then widens to double (exact).  Products of two bf16 values carry at most
 * 16 significant bits and are exact in double; the sum is accumulated in
 * double in k order.
 *
 * Alongside each ref it returns absdot[i][j] = |alpha| * sum_k |a(i,k) b(j,k)|,
 * the quantity the accuracy bound is stated in.
 *
 * If beta == 0, C is not read (it may be NULL).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_C_BF16 0
#define ORACLE_C_F32 1

static double dec_bf16(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double dec_c(const void *C, int64_t idx, int c_dtype) {
  if (c_dtype == ORACLE_C_BF16) return dec_bf16(((const uint16_t *)C)[idx]);
  return (double)((const float *)C)[idx];
}

/* One output element, written out as the definition reads. */
static void one(int64_t i, int64_t j, int64_t K, const uint16_t *A, int64_t lda,
                const uint16_t *B, int64_t ldb, const void *C, int64_t ldc,
                int c_dtype, double alpha, double beta, double *ref,
                double *absdot) {
  double acc = 0.0, mag = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    double p = dec_bf16(A[i * lda + k]) * dec_bf16(B[j * ldb + k]);
    acc += p;
    mag += fabs(p);
  }
  double r = alpha * acc;
  if (beta != 0.0) r += beta * dec_c(C, i * ldc + j, c_dtype);
  *ref = r;
  if (absdot) *absdot = fabs(alpha) * mag;
}

typedef struct {
  int64_t M, N, K, lda, ldb, ldc, ldr;
  const uint16_t *A, *B;
  const void *C;
  int c_dtype;
  double alpha, beta;
  double *ref, *absdot;
  /* sampled mode */
  int64_t nsamples;
  const int64_t *rows, *cols;
  /* work split */
  int64_t begin, end;
} job_t;

static void *run_full(void *p) {
  job_t *j = (job_t *)p;
  for (int64_t i = j->begin; i < j->end; ++i)
    for (int64_t c = 0; c < j->N; ++c)
      one(i, c, j->K, j->A, j->lda, j->B, j->ldb, j->C, j->ldc, j->c_dtype,
          j->alpha, j->beta, &j->ref[i * j->ldr + c],
          j->absdot ? &j->absdot[i * j->ldr + c] : NULL);
  return NULL;
}

static void *run_sampled(void *p) {
  job_t *j = (job_t *)p;
  for (int64_t s = j->begin; s < j->end; ++s)
    one(j->rows[s], j->cols[s], j->K, j->A, j->lda, j->B, j->ldb, j->C, j->ldc,
        j->c_dtype, j->alpha, j->beta, &j->ref[s],
        j->absdot ? &j->absdot[s] : NULL);
  return NULL;
}

static int nthreads_or_default(int nthreads) {
  if (nthreads > 0) return nthreads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static int spawn(job_t base, int64_t total, int nthreads, void *(*fn)(void *)) {
  nthreads = nthreads_or_default(nthreads);
  if (nthreads > total) nthreads = total > 0 ? (int)total : 1;
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
  if (!th || !jobs) {
    free(th);
    free(jobs);
    return -1;
  }
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = base;
    jobs[t].begin = total * t / nthreads;
    jobs[t].end = total * (t + 1) / nthreads;
    if (pthread_create(&th[t], NULL, fn, &jobs[t]) != 0) {
      fn(&jobs[t]); /* run inline if a thread cannot start */
      th[t] = 0;
    }
  }
  for (int t = 0; t < nthreads; ++t)
    if (th[t]) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

/* Full M x N result into ref (and absdot, may be NULL), row stride ldr. */
int oracle_gemm_f64(int64_t M, int64_t N, int64_t K, const uint16_t *A,
                    int64_t lda, const uint16_t *B, int64_t ldb, const void *C,
                    int64_t ldc, int c_dtype, double alpha, double beta,
                    double *ref, double *absdot, int64_t ldr, int nthreads) {
  if (M < 0 || N < 0 || K < 0 || ldr < N) return -1;
  if (beta != 0.0 && C == NULL) return -1;
  job_t b;
  memset(&b, 0, sizeof b);
  b.M = M; b.N = N; b.K = K; b.lda = lda; b.ldb = ldb; b.ldc = ldc; b.ldr = ldr;
  b.A = A; b.B = B; b.C = C; b.c_dtype = c_dtype;
  b.alpha = alpha; b.beta = beta; b.ref = ref; b.absdot = absdot;
  return spawn(b, M, nthreads, run_full);
}

/* ref[s] (and absdot[s]) for the elements (rows[s], cols[s]), s < nsamples. */
int oracle_gemm_f64_sampled(int64_t M, int64_t N, int64_t K, const uint16_t *A,
                            int64_t lda, const uint16_t *B, int64_t ldb,
                            const void *C, int64_t ldc, int c_dtype,
                            double alpha, double beta, int64_t nsamples,
                            const int64_t *rows, const int64_t *cols,
                            double *ref, double *absdot, int nthreads) {
  if (M < 0 || N < 0 || K < 0 || nsamples < 0) return -1;
  if (beta != 0.0 && C == NULL) return -1;
  for (int64_t s = 0; s < nsamples; ++s)
    if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return -1;
  job_t b;
  memset(&b, 0, sizeof b);
  b.M = M; b.N = N; b.K = K; b.lda = lda; b.ldb = ldb; b.ldc = ldc;
  b.A = A; b.B = B; b.C = C; b.c_dtype = c_dtype;
  b.alpha = alpha; b.beta = beta; b.ref = ref; b.absdot = absdot;
  b.nsamples = nsamples; b.rows = rows; b.cols = cols;
  return spawn(b, nsamples, nthreads, run_sampled);
}

int oracle_nthreads_default(void) { return nthreads_or_default(0); }

/*
 * FP8 operands.  A one-byte value decodes by its format's definition:
 *   e4m3 (fmt 0): sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent
 *     field 0 is subnormal (2^-6 * m/8); all-ones exponent with mantissa 7 is
 *     NaN, the other all-ones codes are finite (max 448); no infinities.
 *   e5m2 (fmt 1): sign, 5 exponent bits (bias 15), 2 mantissa bits; exponent
 *     field 0 is subnormal (2^-14 * m/4); all-ones exponent is infinity
 *     (mantissa 0) or NaN.
 * Products of two fp8 values are exact in double, as is their k-order sum
 * for the sizes used here.
 */
static double dec_fp8(uint8_t v, int fmt) {
  const int s = v >> 7;
  double x;
  if (fmt == 0) {
    const int e = (v >> 3) & 0xF, m = v & 7;
    if (e == 0xF && m == 7) x = NAN;
    else if (e == 0) x = ldexp((double)m / 8.0, -6);
    else x = ldexp(1.0 + (double)m / 8.0, e - 7);
  } else {
    const int e = (v >> 2) & 0x1F, m = v & 3;
    if (e == 0x1F) x = m == 0 ? INFINITY : NAN;
    else if (e == 0) x = ldexp((double)m / 4.0, -14);
    else x = ldexp(1.0 + (double)m / 4.0, e - 15);
  }
  return s ? -x : x;
}

typedef struct {
  int64_t N, K, lda, ldb, ldc, ldr;
  const uint8_t *A, *B;
  int fmt;
  const void *C;
  int c_dtype;
  double alpha, beta;
  double *ref, *absdot;
  const int64_t *rows, *cols; /* sampled mode when non-NULL */
  int64_t begin, end;
} job8_t;

/* One output element, D[i][c] in FP64, and sum |alpha a_ik b_ck| beside it. */
static void one_fp8(const job8_t *j, int64_t i, int64_t c, double *ref, double *absdot) {
  double acc = 0.0, mag = 0.0;
  for (int64_t k = 0; k < j->K; ++k) {
    double pr = dec_fp8(j->A[i * j->lda + k], j->fmt) * dec_fp8(j->B[c * j->ldb + k], j->fmt);
    acc += pr;
    mag += fabs(pr);
  }
  double r = j->alpha * acc;
  if (j->beta != 0.0) r += j->beta * dec_c(j->C, i * j->ldc + c, j->c_dtype);
  *ref = r;
  if (absdot) *absdot = fabs(j->alpha) * mag;
}

static void *run_fp8(void *p) {
  job8_t *j = (job8_t *)p;
  if (j->rows) {
    for (int64_t s = j->begin; s < j->end; ++s)
      one_fp8(j, j->rows[s], j->cols[s], &j->ref[s], j->absdot ? &j->absdot[s] : NULL);
    return NULL;
  }
  for (int64_t i = j->begin; i < j->end; ++i)
    for (int64_t c = 0; c < j->N; ++c)
      one_fp8(j, i, c, &j->ref[i * j->ldr + c], j->absdot ? &j->absdot[i * j->ldr + c] : NULL);
  return NULL;
}

static int spawn_fp8(job8_t base, int64_t total, int nthreads) {
  nthreads = nthreads_or_default(nthreads);
  if (nthreads > total) nthreads = total > 0 ? (int)total : 1;
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  job8_t *jobs = (job8_t *)calloc((size_t)nthreads, sizeof(job8_t));
  if (!th || !jobs) {
    free(th);
    free(jobs);
    return -1;
  }
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = base;
    jobs[t].begin = total * t / nthreads;
    jobs[t].end = total * (t + 1) / nthreads;
    if (pthread_create(&th[t], NULL, run_fp8, &jobs[t]) != 0) {
      run_fp8(&jobs[t]);
      th[t] = 0;
    }
  }
  for (int t = 0; t < nthreads; ++t)
    if (th[t]) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

/* Full FP64 reference for fp8 A (M x lda bytes) and B (N x ldb bytes). */
int oracle_gemm_fp8_f64(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B,
                        int64_t ldb, int fmt, const void *C, int64_t ldc, int c_dtype, double alpha,
                        double beta, double *ref, double *absdot, int64_t ldr, int nthreads) {
  if (M < 0 || N < 0 || K < 0 || ldr < N || (fmt != 0 && fmt != 1)) return -1;
  if (beta != 0.0 && C == NULL) return -1;
  job8_t b = {N, K, lda, ldb, ldc, ldr, A, B, fmt, C, c_dtype, alpha, beta, ref, absdot, NULL, NULL, 0, 0};
  return spawn_fp8(b, M, nthreads);
}

/* The same at the listed (rows[s], cols[s]) only; ref and absdot hold nsamples values. */
int oracle_gemm_fp8_f64_sampled(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda,
                                const uint8_t *B, int64_t ldb, int fmt, const void *C, int64_t ldc,
                                int c_dtype, double alpha, double beta, int64_t nsamples,
                                const int64_t *rows, const int64_t *cols, double *ref, double *absdot,
                                int nthreads) {
  if (M < 0 || N < 0 || K < 0 || nsamples < 0 || (fmt != 0 && fmt != 1)) return -1;
  if (beta != 0.0 && C == NULL) return -1;
  for (int64_t s = 0; s < nsamples; ++s)
    if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return -1;
  job8_t b = {N, K, lda, ldb, ldc, 0, A, B, fmt, C, c_dtype, alpha, beta, ref, absdot, rows, cols, 0, 0};
  return spawn_fp8(b, nsamples, nthreads);
}

/*
 * Fused MLP epilogue, in FP64: ref[i][j] <- act(ref[i][j] + bias[j]).
 *
 * bias holds N values (bf16 bits, bias_dtype 0, or float, bias_dtype 1) or
 * is NULL.  act: 0 none, 1 ReLU max(x, 0), 2 GELU x * Phi(x) with
 * Phi(x) = (1 + erf(x / sqrt 2)) / 2, 3 the tanh approximation of GELU
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), 4 SiLU x / (1 + e^-x).
 * These are the usual definitions of the activations an MLP up-projection
 * applies after adding its bias (the epilogue-fusion step the H100 Nsight
 * Compute page lists among GEMM optimisations, section 7).
 */
static double act_f64(double x, int act) {
  switch (act) {
    case 1: return x > 0.0 ? x : 0.0;
    case 2: return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
    case 3: {
      const double k = sqrt(2.0 / 3.14159265358979323846);
      return 0.5 * x * (1.0 + tanh(k * (x + 0.044715 * x * x * x)));
    }
    case 4: return x / (1.0 + exp(-x));
    default: return x;
  }
}

int oracle_epilogue_f64(int64_t M, int64_t N, double *ref, int64_t ldr,
                        const void *bias, int bias_dtype, int act) {
  if (M < 0 || N < 0 || ldr < N || act < 0 || act > 4) return -1;
  for (int64_t i = 0; i < M; ++i)
    for (int64_t j = 0; j < N; ++j) {
      double b = 0.0;
      if (bias) b = bias_dtype == 0 ? dec_bf16(((const uint16_t *)bias)[j]) : (double)((const float *)bias)[j];
      ref[i * ldr + j] = act_f64(ref[i * ldr + j] + b, act);
    }
  return 0;
}
