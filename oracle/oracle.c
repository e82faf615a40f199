/*
 * CPU oracle for the autotuned dense matmul.  TEST INFRASTRUCTURE ONLY: the
 * library never links, loads or calls this file; only the tests, the bench's
 * CPU-baseline leg and the smoke check do.
 *
 * What it computes.  Every candidate kernel of the tuner computes the same
 * mathematical object, C = A.B; configurations change how the sum is formed,
 * not what it is (CMU 15-779 Lecture 9, section 2.1: "configs only change how,
 * not what", shown there on split-K).  The oracle is therefore the plain
 * definition
 *
 *     C[b][i][j] = sum_{k < K} A[b][i][k] * B[b][k][j]
 *
 * accumulated in IEEE binary64 in increasing k, one output at a time, with
 * A and B read through arbitrary element strides so that transposed views are
 * read in place (burn "cubecl-backend" page, section "matmul: handing strides
 * to cubek": the matmul gets strides and never makes its inputs contiguous).
 *
 * Rounding of the result to the output type is a separate step, written from
 * the IEEE 754 definitions: binary32 by the C cast (round to nearest, ties to
 * even, in the default rounding mode), bfloat16 and binary16 by an explicit
 * nearest-even rounding to the format's precision with its subnormals and
 * overflow to infinity.
 *
 * The only parallelism is an OpenMP loop over output rows; nothing is blocked,
 * fused or reordered.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_F16 = 1, ORC_F32 = 2 };

/* bfloat16: the top 16 bits of a binary32. */
static double orc_from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double orc_from_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(f + 1024), e - 25); /* (1 + f/1024) * 2^(e-15) */
  return sign ? -v : v;
}

static double orc_load(const void *base, int64_t idx, int dtype) {
  switch (dtype) {
  case ORC_BF16: return orc_from_bf16(((const uint16_t *)base)[idx]);
  case ORC_F16: return orc_from_f16(((const uint16_t *)base)[idx]);
  default: return (double)((const float *)base)[idx];
  }
}

/*
 * C64[b*M*N + i*N + j] = sum_k A(b,i,k) * B(b,k,j) in binary64, k ascending.
 * Element (b,i,k) of A is at a_bs*b + a_rs*i + a_cs*k (elements), likewise B.
 */
void oracle_gemm_f64(const void *A, int dtA, int64_t a_rs, int64_t a_cs, int64_t a_bs,
                     const void *B, int dtB, int64_t b_rs, int64_t b_cs, int64_t b_bs,
                     double *C64, int64_t M, int64_t N, int64_t K, int64_t batch) {
  int64_t rows = batch * M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < rows; ++r) {
    int64_t b = r / (M ? M : 1), i = r % (M ? M : 1);
    for (int64_t j = 0; j < N; ++j) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += orc_load(A, b * a_bs + i * a_rs + k * a_cs, dtA) *
               orc_load(B, b * b_bs + k * b_rs + j * b_cs, dtB);
      C64[(b * M + i) * N + j] = acc;
    }
  }
}

/* The same sum for a list of (b, i, j) points; out[p] for point p. */
void oracle_gemm_points(const void *A, int dtA, int64_t a_rs, int64_t a_cs, int64_t a_bs,
                        const void *B, int dtB, int64_t b_rs, int64_t b_cs, int64_t b_bs,
                        int64_t K, const int64_t *bij, int64_t npoints, double *out) {
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < npoints; ++p) {
    int64_t b = bij[3 * p], i = bij[3 * p + 1], j = bij[3 * p + 2];
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
      acc += orc_load(A, b * a_bs + i * a_rs + k * a_cs, dtA) *
             orc_load(B, b * b_bs + k * b_rs + j * b_cs, dtB);
    out[p] = acc;
  }
}

/*
 * Round a binary64 value to a binary format with `p` significand bits
 * (including the implicit one), minimum normal exponent `emin` and maximum
 * finite value `maxv`, to nearest with ties to even.  Returns the rounded
 * value as a double (exact).  Follows IEEE 754: the representable numbers
 * below 2^emin are the multiples of 2^(emin-p+1) (subnormals); values whose
 * rounded magnitude exceeds maxv become infinity.
 */
static double orc_round_to_format(double x, int p, int emin, double maxv) {
  if (isnan(x) || isinf(x) || x == 0.0)
    return x;
  double ax = fabs(x);
  int e;
  frexp(ax, &e);      /* ax = f * 2^e with f in [0.5, 1): exponent of ax is e-1 */
  int ex = e - 1;
  if (ex < emin)
    ex = emin;        /* subnormal range: fixed quantum */
  double quantum = ldexp(1.0, ex - (p - 1));
  double q = ax / quantum;              /* exact: power-of-two scaling */
  double fl = floor(q);
  double rem = q - fl;
  double r;
  if (rem > 0.5)
    r = fl + 1.0;
  else if (rem < 0.5)
    r = fl;
  else
    r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0; /* tie: to even */
  double v = r * quantum;
  if (v > maxv)
    v = INFINITY;
  return x < 0 ? -v : v;
}

/* bfloat16: p = 8, emin = -126, max = (2 - 2^-7) * 2^127. */
void oracle_round_bf16(const double *x, uint16_t *out, int64_t n) {
  const double maxv = ldexp(255.0, 120);
  for (int64_t t = 0; t < n; ++t) {
    double v = orc_round_to_format(x[t], 8, -126, maxv);
    float f = (float)v;  /* exact: v is representable in binary32 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(x[t]))
      u = 0x7FC00000u;
    out[t] = (uint16_t)(u >> 16);
  }
}

/* binary16: p = 11, emin = -14, max = 65504. */
void oracle_round_f16(const double *x, uint16_t *out, int64_t n) {
  for (int64_t t = 0; t < n; ++t) {
    double xv = x[t];
    uint16_t h;
    if (isnan(xv)) {
      h = 0x7E00;
    } else {
      double v = orc_round_to_format(xv, 11, -14, 65504.0);
      uint16_t s = (v < 0 || (v == 0 && signbit(v))) ? 0x8000 : 0;
      double a = fabs(v);
      if (isinf(a)) {
        h = s | 0x7C00;
      } else if (a < ldexp(1.0, -14)) {
        h = s | (uint16_t)(a / ldexp(1.0, -24)); /* subnormal: exact multiple */
      } else {
        int e;
        double f = frexp(a, &e);  /* a = f*2^e, f in [0.5,1) */
        int biased = e - 1 + 15;
        uint16_t frac = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
        h = s | (uint16_t)(biased << 10) | frac;
      }
    }
    out[t] = h;
  }
}

/* binary32: the C conversion rounds to nearest, ties to even. */
void oracle_round_f32(const double *x, float *out, int64_t n) {
  for (int64_t t = 0; t < n; ++t)
    out[t] = (float)x[t];
}

/* Threads the OpenMP runtime will use for the loops above. */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Use n threads (n >= 1) for the loops above from now on; for timing the
 * oracle on one core beside all of them.  No effect without OpenMP. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
