/*
 * fp8_oracle.c -- plain, slow CPU oracle for the per-tensor scaled FP8 linear path.
 *
 * TEST INFRASTRUCTURE ONLY: used by tests, the smoke check and the benchmark's
 * CPU-baseline leg; never by the product path.  Shares no source with the CUDA
 * library.  See fp8_oracle.h for the page references ([TE], [LP]).
 *
 * Readings of the pages taken here (the pages leave these open):
 *  - Bit layouts and special values follow OCP FP8, the standard [TE] S4.2.8
 *    names:  E4M3 = bias 7, no Inf, S.1111.111 is NaN, largest finite 0x7E = 448;
 *    E5M2 = bias 15, IEEE-style Inf/NaN, largest finite 0x7B = 57344.
 *  - "round_to_fp8" ([TE] S4.2.4) is round-to-nearest, ties to even mantissa, and
 *    magnitudes above FP8_MAX (Inf included) saturate to +-FP8_MAX ([TE] S4.2.4
 *    describes overflow of too small a scale as saturation).
 *  - NaN encodes to 0x7F (E4M3) / 0x7E (E5M2).
 *  - "tensor x scale" is an fp32 product rounded to nearest, then one FP8 rounding.
 *  - scale = FP8_MAX / amax is an fp32 IEEE division with no margin; a zero or
 *    non-finite amax keeps the previous scale; an overflowing quotient is clamped
 *    to FLT_MAX.
 *
 * Compile with -ffp-contract=off so that no multiply-add is fused.
 */
#include "fp8_oracle.h"

#include <float.h>
#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Formats ([TE] S4.2.3: E4M3 = 4 exponent / 3 mantissa bits, E5M2 = 5 / 2).  */
/* ------------------------------------------------------------------------- */

double oracle_fp8_decode(uint8_t code, int fmt) {
  const double sign = (code & 0x80) ? -1.0 : 1.0;
  if (fmt == ORACLE_E4M3) {
    const int e = (code >> 3) & 0xF;
    const int f = code & 0x7;
    if (e == 0xF && f == 0x7) return NAN;                 /* S.1111.111 */
    if (e == 0) return sign * ldexp((double)f, -9);        /* f/8 * 2^(1-7) */
    return sign * ldexp(1.0 + f / 8.0, e - 7);             /* (1+f/8) * 2^(e-7) */
  } else {
    const int e = (code >> 2) & 0x1F;
    const int f = code & 0x3;
    if (e == 0x1F) return (f == 0) ? sign * INFINITY : NAN;
    if (e == 0) return sign * ldexp((double)f, -16);       /* f/4 * 2^(1-15) */
    return sign * ldexp(1.0 + f / 4.0, e - 15);            /* (1+f/4) * 2^(e-15) */
  }
}

static int top_code(int fmt) { return fmt == ORACLE_E4M3 ? 0x7E : 0x7B; }

double oracle_fp8_max(int fmt) { return oracle_fp8_decode((uint8_t)top_code(fmt), fmt); }

/* Non-negative finite code values, ascending in code order, filled once from
 * oracle_fp8_decode so that the encoder searches exactly the decoded set. */
static double g_table[2][128];
__attribute__((constructor)) static void oracle_init_tables(void) {
  for (int fmt = 0; fmt < 2; ++fmt)
    for (int c = 0; c <= top_code(fmt); ++c) g_table[fmt][c] = oracle_fp8_decode((uint8_t)c, fmt);
}

uint8_t oracle_fp8_encode_double(double v, int fmt) {
  if (isnan(v)) return fmt == ORACLE_E4M3 ? 0x7F : 0x7E;
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs(v);
  const int top = top_code(fmt);
  const double* t = g_table[fmt];
  if (a > t[top]) return (uint8_t)(sign | top); /* saturate, Inf included */
  /* largest code c with value(c) <= a (values ascend with the code) */
  int lo = 0, hi = top;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (t[mid] <= a) lo = mid; else hi = mid - 1;
  }
  const int c = lo;
  if (c == top || t[c] == a) return (uint8_t)(sign | c);
  /* a lies strictly between value(c) and value(c+1); their midpoint is exact in
   * double, so this compare is exact. */
  const double midpoint = 0.5 * (t[c] + t[c + 1]);
  if (a < midpoint) return (uint8_t)(sign | c);
  if (a > midpoint) return (uint8_t)(sign | (c + 1));
  return (uint8_t)(sign | ((c & 1) ? c + 1 : c)); /* tie: even mantissa LSB */
}

uint8_t oracle_fp8_encode(float v, int fmt) { return oracle_fp8_encode_double((double)v, fmt); }

void oracle_fp8_decode_array(const uint8_t* codes, int64_t n, int fmt, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp8_decode(codes[i], fmt);
}

void oracle_fp8_encode_array(const float* v, int64_t n, int fmt, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp8_encode(v[i], fmt);
}

/* ------------------------------------------------------------------------- */
/* bf16                                                                       */
/* ------------------------------------------------------------------------- */

float oracle_bf16_to_float(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16; /* bf16 is the top half of an fp32 */
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round a double to the nearest bf16 (8-bit significand, fp32 exponent range),
 * ties to even; overflow past the rounding boundary gives +-Inf. */
uint16_t oracle_double_to_bf16(double y) {
  if (isnan(y)) return 0x7FC0;
  const uint16_t sign = signbit(y) ? 0x8000 : 0x0000;
  const double a = fabs(y);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e2;
  frexp(a, &e2);               /* a = m * 2^e2, m in [0.5, 1) */
  int E = e2 - 1;              /* floor(log2 a) */
  if (E < -126) E = -126;      /* subnormal range shares the quantum 2^-133 */
  const double quantum = ldexp(1.0, E - 7);
  const double r = nearbyint(a / quantum); /* a/quantum is exact; default mode = ties-to-even */
  const double v = r * quantum;
  if (v >= 0x1p128) return (uint16_t)(sign | 0x7F80);
  const float f = (float)v; /* exact: v has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (u >> 16));
}

void oracle_double_to_bf16_array(const double* y, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_bf16(y[i]);
}

/* ------------------------------------------------------------------------- */
/* amax, scale, cast ([TE] S4.2.4)                                            */
/* ------------------------------------------------------------------------- */

float oracle_amax_bf16(const uint16_t* x, int64_t n) {
  float m = 0.0f;
  int saw_nan = 0;
#pragma omp parallel for schedule(static) reduction(max : m) reduction(| : saw_nan)
  for (int64_t i = 0; i < n; ++i) {
    const float a = fabsf(oracle_bf16_to_float(x[i]));
    if (isnan(a)) saw_nan = 1;
    else if (a > m) m = a;
  }
  return saw_nan ? NAN : m;
}

void oracle_cast_bf16(const uint16_t* x, int64_t n, float scale, int fmt, uint8_t* q,
                      uint64_t* n_sat, uint64_t* n_und) {
  const float fmax = (float)oracle_fp8_max(fmt);
  uint64_t sat = 0, und = 0;
#pragma omp parallel for schedule(static) reduction(+ : sat, und)
  for (int64_t i = 0; i < n; ++i) {
    const float xf = oracle_bf16_to_float(x[i]);
    const float p = xf * scale; /* fp32, round to nearest */
    const uint8_t c = oracle_fp8_encode(p, fmt);
    q[i] = c;
    if (fabsf(p) > fmax) ++sat;                      /* clipped by saturation */
    if (xf != 0.0f && (c & 0x7F) == 0) ++und;        /* nonzero flushed to +-0 */
  }
  *n_sat = sat;
  *n_und = und;
}

float oracle_scale_from_amax(float m, int fmt, float prev_scale) {
  if (!(m > 0.0f) || isinf(m)) return prev_scale; /* zero, NaN or Inf: keep */
  float s = (float)oracle_fp8_max(fmt) / m;      /* fp32 IEEE division */
  if (isinf(s)) s = FLT_MAX;
  return s;
}

float oracle_reciprocal(float s) { return 1.0f / s; }

/* ------------------------------------------------------------------------- */
/* GEMM ([TE] S4.2.4: FP8 multiply, FP32-or-wider accumulation, x(1/scale)).   */
/* ------------------------------------------------------------------------- */

void oracle_gemm_rows(const uint8_t* A, int afmt, int64_t lda, const uint8_t* B, int bfmt,
                      int64_t ldb, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                      int64_t nrows, float factor, double* acc, double* absacc, uint16_t* out) {
  (void)M;
  double da[256], db[256];
  for (int c = 0; c < 256; ++c) {
    da[c] = oracle_fp8_decode((uint8_t)c, afmt);
    db[c] = oracle_fp8_decode((uint8_t)c, bfmt);
  }
  const int64_t count = rows ? nrows : M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < count; ++i) {
    const int64_t r = rows ? rows[i] : i;
    const uint8_t* a = A + r * lda;
    for (int64_t n = 0; n < N; ++n) {
      const uint8_t* b = B + n * ldb;
      double s = 0.0, sa = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double prod = da[a[k]] * db[b[k]]; /* exact: 4x4 / 3x3 significand bits */
        s += prod;
        sa += fabs(prod);
      }
      acc[i * N + n] = s;
      if (absacc) absacc[i * N + n] = sa;
      if (out) out[i * N + n] = oracle_double_to_bf16(s * (double)factor);
    }
  }
}

/* ------------------------------------------------------------------------- */
/* Block scaling, MX style ([LP] format overview: per-tensor *or per-block*     */
/* scale factors; MXFP8 = FP8 elements that share one scale per small block).   */
/* ------------------------------------------------------------------------- */
/* Readings (the pages name the formats but give no rule):
 *  - a block is 32 consecutive elements of a row (the last block of a row may be
 *    shorter); its scale is a power of two 2^-k stored as an E8M0 code 127 - k;
 *  - k follows the per-tensor rule "scale = FP8_MAX / amax" restricted to powers
 *    of two: the largest k in [-127, 127] with amax_block * 2^k <= FP8_MAX, so
 *    that no element saturates; -127 when there is none (an Inf or NaN amax);
 *  - element code = round_to_fp8(x * 2^k), exact product, one RNE rounding. */

int oracle_mx_scale_exponent(double amax, int fmt) {
  const double fmax = oracle_fp8_max(fmt);
  for (int k = 127; k >= -127; --k)
    if (ldexp(amax, k) <= fmax) return k; /* exact: amax is a bf16 value */
  return -127;
}

double oracle_e8m0_value(uint8_t code) { return code == 0xFF ? NAN : ldexp(1.0, (int)code - 127); }

void oracle_mx_quantize(const uint16_t* x, int64_t rows, int64_t cols, int fmt, uint8_t* q,
                        uint8_t* scale) {
  const int64_t nb = (cols + 31) / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const int64_t c0 = 32 * b;
      const int64_t c1 = c0 + 32 < cols ? c0 + 32 : cols;
      double amax = 0.0;
      int nan = 0;
      for (int64_t c = c0; c < c1; ++c) {
        const double a = fabs((double)oracle_bf16_to_float(x[r * cols + c]));
        if (isnan(a)) nan = 1;
        else if (a > amax) amax = a;
      }
      const int k = oracle_mx_scale_exponent(nan ? NAN : amax, fmt);
      scale[r * nb + b] = (uint8_t)(127 - k);
      for (int64_t c = c0; c < c1; ++c)
        q[r * cols + c] = oracle_fp8_encode_double(ldexp((double)oracle_bf16_to_float(x[r * cols + c]), k), fmt);
    }
  }
}

void oracle_mx_gemm_rows(const uint8_t* A, int afmt, const uint8_t* sa, const uint8_t* B, int bfmt,
                         const uint8_t* sb, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                         int64_t nrows, double* acc, double* absacc, uint16_t* out) {
  double da[256], db[256];
  for (int c = 0; c < 256; ++c) {
    da[c] = oracle_fp8_decode((uint8_t)c, afmt);
    db[c] = oracle_fp8_decode((uint8_t)c, bfmt);
  }
  const int64_t nb = (K + 31) / 32;
  const int64_t count = rows ? nrows : M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < count; ++i) {
    const int64_t r = rows ? rows[i] : i;
    const uint8_t* a = A + r * K;
    for (int64_t n = 0; n < N; ++n) {
      const uint8_t* b = B + n * K;
      double s = 0.0, sabs = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        /* dequantised operands: element value times its block's scale (exact) */
        const double av = da[a[k]] * oracle_e8m0_value(sa[r * nb + k / 32]);
        const double bv = db[b[k]] * oracle_e8m0_value(sb[n * nb + k / 32]);
        s += av * bv;
        sabs += fabs(av * bv);
      }
      acc[i * N + n] = s;
      if (absacc) absacc[i * N + n] = sabs;
      if (out) out[i * N + n] = oracle_double_to_bf16(s);
    }
  }
}

/* ------------------------------------------------------------------------- */
/* FP8 gradient all-reduce with automatic scaling.                            */
/* [LP] use cases: E5M2 for gradient communication in distributed training, to */
/* cut inter-node bandwidth.  [FL] (forum thread on the FP8-LM paper):          */
/* "automatic scaling" adjusts the tensor scaling factor dynamically so that    */
/* gradients stay inside FP8's range during the all-reduce.                     */
/* ------------------------------------------------------------------------- */
/* Readings: the ranks agree on amax = max over all ranks of max|g|, and on one
 * scale s = 57344 / (world * amax) in fp32 (world * amax an fp32 product,
 * clamped to FLT_MAX; s = 1 when amax is 0 or not finite; an overflowing
 * quotient is clamped to FLT_MAX), so that the world-way sum of the scaled
 * values cannot leave E5M2's range; every rank casts fp32(g * s) to E5M2; the
 * codes are summed exactly and the sum is rounded once more to E5M2 (RNE,
 * saturating) -- the value that travels; the result is
 * bf16(fp32(decode(sum code) * f)) with f = 1/s (sum) or fp32((1/s) / world)
 * (mean). */

float oracle_allreduce_scale(float amax, int world) {
  if (!(amax > 0.0f) || isinf(amax)) return 1.0f;
  float d = (float)world * amax; /* fp32 product */
  if (isinf(d)) d = FLT_MAX;
  float s = 57344.0f / d;        /* fp32 division */
  if (isinf(s)) s = FLT_MAX;
  return s;
}

void oracle_allreduce_e5m2(const uint16_t* g, int world, int64_t n, int average, uint16_t* out,
                           uint8_t* codes, float* scale) {
  const float amax = oracle_amax_bf16(g, (int64_t)world * n);
  const float s = oracle_allreduce_scale(amax, world);
  const float sinv = 1.0f / s;
  const float f = average ? sinv / (float)world : sinv;
  if (scale) {
    scale[0] = s;
    scale[1] = sinv;
  }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double sum = 0.0; /* exact: at most 32 + log2(world) significant bits */
    for (int r = 0; r < world; ++r) {
      const float p = oracle_bf16_to_float(g[(int64_t)r * n + i]) * s; /* fp32 product */
      sum += oracle_fp8_decode(oracle_fp8_encode(p, ORACLE_E5M2), ORACLE_E5M2);
    }
    const uint8_t c = oracle_fp8_encode_double(sum, ORACLE_E5M2);
    if (codes) codes[i] = c;
    const float y = (float)oracle_fp8_decode(c, ORACLE_E5M2) * f; /* exact decode, fp32 product */
    out[i] = oracle_double_to_bf16((double)y);
  }
}

/* ------------------------------------------------------------------------- */
/* Epilogue cast and the MLP activation (the transformer layer of [TE] S4.2.6).  */
/* ------------------------------------------------------------------------- */

void oracle_cast_f32(const float* v, int64_t n, float scale, int fmt, uint8_t* q, uint64_t* n_sat,
                     uint64_t* n_und, float* amax) {
  const float fmax = (float)oracle_fp8_max(fmt);
  uint64_t sat = 0, und = 0;
  float m = 0.0f;
  int saw_nan = 0;
#pragma omp parallel for schedule(static) reduction(+ : sat, und) reduction(max : m) reduction(| : saw_nan)
  for (int64_t i = 0; i < n; ++i) {
    const float p = v[i] * scale; /* fp32, round to nearest */
    const uint8_t c = oracle_fp8_encode(p, fmt);
    q[i] = c;
    if (fabsf(p) > fmax) ++sat;
    if (v[i] != 0.0f && (c & 0x7F) == 0) ++und;
    const float a = fabsf(v[i]);
    if (isnan(a)) saw_nan = 1;
    else if (a > m) m = a;
  }
  *n_sat = sat;
  *n_und = und;
  *amax = saw_nan ? NAN : m;
}

/* tanh form of GELU: x * Phi(x) with the normal CDF replaced by
 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))) / 2. */
static const double kGeluA = 0.044715;

static double gelu_c(void) { return sqrt(2.0 / (4.0 * atan(1.0))); } /* sqrt(2/pi) */

double oracle_gelu(double x) {
  const double c = gelu_c();
  const double t = tanh(c * (x + kGeluA * x * x * x));
  return 0.5 * x * (1.0 + t);
}

/* Product rule on x/2 * (1 + t(x)), with t' = (1 - t^2) * c * (1 + 3a x^2). */
double oracle_dgelu(double x) {
  const double c = gelu_c();
  const double t = tanh(c * (x + kGeluA * x * x * x));
  const double dt = (1.0 - t * t) * c * (1.0 + 3.0 * kGeluA * x * x);
  return 0.5 * (1.0 + t) + 0.5 * x * dt;
}

void oracle_gelu_array(const double* x, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_gelu(x[i]);
}

void oracle_dgelu_array(const double* x, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_dgelu(x[i]);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads of the calling thread's later parallel regions (n >= 1); a no-op
   without OpenMP.  Changes no result: every parallel loop here writes
   disjoint outputs, and its reductions (max, bitwise or, integer counts) give
   the same value in any order. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
