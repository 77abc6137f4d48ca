/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU restatement of the matrix products of a
 * linear layer in a training step, evaluated in fp64.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load this code; the
 * library's product path never does.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Source of the definition: "Twice the training speed on a BC-250 from tuned
 * matrix kernels", section "Checking the results are right": every product
 * (FP32, fp16 and bf16 inputs, all three layouts, batched attention) is
 * compared with a float64 product computed on the CPU.  Section "Where the
 * time went" defines the three products of a linear layer (forward, input
 * gradient, weight gradient) and section "Tuning the kernels" fixes FP32
 * accumulation over 16-bit inputs.  Tuning changes no arithmetic, so the
 * exact product of the rounded inputs is the oracle:
 *
 *     C[b,i,j] = sum_{k=0}^{K-1} A(b,i,k) * B(b,k,j)      (fp64, k ascending)
 *     S[b,i,j] = sum_{k=0}^{K-1} |A(b,i,k) * B(b,k,j)|    (error scale)
 *
 * Every operand is addressed through explicit element strides, so each of the
 * layer's layouts is this one loop nest with its own index map (the maps live
 * in oracle/__init__.py).  16-bit inputs are decoded exactly (every bf16 and
 * fp16 value is a double).  There is no blocking, no fusion and no reordering:
 * one dot product per output element, k ascending.  Threads (OpenMP) split
 * output rows only, so results do not depend on the thread count.
 *
 * The header of oracle/__init__.py lists what pins each function.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element types: identical numbering to the Python side of the oracle */
enum { OR_BF16 = 0, OR_F16 = 1, OR_F32 = 2, OR_F64 = 3 };

/* bf16: the upper half of an IEEE binary32 */
static double dec_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* fp16 (IEEE binary16): 1 sign, 5 exponent (bias 15), 10 fraction bits */
static double dec_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

static double load(const void *p, int dt, int64_t idx) {
  switch (dt) {
  case OR_BF16: return dec_bf16(((const uint16_t *)p)[idx]);
  case OR_F16: return dec_f16(((const uint16_t *)p)[idx]);
  case OR_F32: return (double)((const float *)p)[idx];
  default: return ((const double *)p)[idx];
  }
}

int oracle_version(void) { return 1; }

/* Decode n 16/32/64-bit values to doubles (exact). */
void oracle_decode(const void *src, int dt, int64_t n, double *dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = load(src, dt, i);
}

/*
 * The product.  A(b,i,k) = A[b*a_bs + i*a_rs + k*a_cs], likewise B(b,k,j).
 * C and S are dense [batch][M][N] doubles; S may be NULL.
 */
void oracle_gemm(const void *A, int adt, int64_t a_bs, int64_t a_rs, int64_t a_cs,
                 const void *B, int bdt, int64_t b_bs, int64_t b_rs, int64_t b_cs,
                 int64_t batch, int64_t M, int64_t N, int64_t K,
                 double *C, double *S, int nthreads) {
  int64_t rows = batch * M;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t r = 0; r < rows; ++r) {
    int64_t b = r / M, i = r % M;
    for (int64_t j = 0; j < N; ++j) {
      double c = 0.0, s = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = load(A, adt, b * a_bs + i * a_rs + k * a_cs) *
                   load(B, bdt, b * b_bs + k * b_rs + j * b_cs);
        c += p;
        s += fabs(p);
      }
      C[r * N + j] = c;
      if (S) S[r * N + j] = s;
    }
  }
  (void)nthreads;
}

/*
 * The same product at n chosen output coordinates (bi[t], ii[t], jj[t]):
 * one fp64 dot product of length K per sample, identical to oracle_gemm's.
 */
void oracle_gemm_at(const void *A, int adt, int64_t a_bs, int64_t a_rs, int64_t a_cs,
                    const void *B, int bdt, int64_t b_bs, int64_t b_rs, int64_t b_cs,
                    int64_t K, int64_t n, const int64_t *bi, const int64_t *ii,
                    const int64_t *jj, double *C, double *S, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
#endif
  for (int64_t t = 0; t < n; ++t) {
    double c = 0.0, s = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double p = load(A, adt, bi[t] * a_bs + ii[t] * a_rs + k * a_cs) *
                 load(B, bdt, bi[t] * b_bs + k * b_rs + jj[t] * b_cs);
      c += p;
      s += fabs(p);
    }
    C[t] = c;
    if (S) S[t] = s;
  }
  (void)nthreads;
}

/*
 * Round-to-nearest-even from a double straight to bf16 or fp16 (no detour
 * through binary32, so no double rounding).  A format with p significant bits,
 * minimum normal exponent emin and maximum exponent emax represents values on
 * the grid q = 2^(max(e, emin) - (p-1)) where e = floor(log2|x|); rint() in
 * the default rounding mode rounds x/q to the nearest integer, ties to even.
 * Overflow goes to infinity; subnormals are kept (not flushed).
 */
static uint16_t rne16(double x, int p, int emin, int emax, int ebits) {
  int fbits = p - 1;
  uint16_t sign = signbit(x) ? (uint16_t)(1u << 15) : 0;
  uint16_t expmask = (uint16_t)(((1u << ebits) - 1) << fbits);
  if (isnan(x)) return (uint16_t)(expmask | (1u << (fbits - 1)));
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | expmask);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): floor(log2 a) = e - 1 */
  int eq = e - 1;
  if (eq < emin) eq = emin;
  double q = ldexp(1.0, eq - fbits);
  double n = rint(a / q); /* integer count of quanta, ties to even */
  double v = n * q;
  if (v == 0.0) return sign; /* rounded down to a signed zero */
  if (v >= ldexp(1.0, emax + 1)) return (uint16_t)(sign | expmask);
  (void)frexp(v, &e);
  int ev = e - 1;
  if (ev < emin) { /* subnormal: exponent field 0, fraction = v / 2^(emin - fbits) */
    uint32_t frac = (uint32_t)ldexp(v, fbits - emin);
    return (uint16_t)(sign | frac);
  }
  int bias = (1 << (ebits - 1)) - 1;
  uint32_t frac = (uint32_t)(ldexp(v, fbits - ev) - ldexp(1.0, fbits));
  return (uint16_t)(sign | ((uint32_t)(ev + bias) << fbits) | frac);
}

/* dt: OR_BF16 (p=8, emin=-126, emax=127) or OR_F16 (p=11, emin=-14, emax=15) */
void oracle_round16(const double *x, int64_t n, int dt, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = dt == OR_BF16 ? rne16(x[i], 8, -126, 127, 8) : rne16(x[i], 11, -14, 15, 5);
}

/* RNE from double to binary32 is what the C cast does in the default mode. */
void oracle_round32(const double *x, int64_t n, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (float)x[i];
}
