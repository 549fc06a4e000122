/*
 * i8_oracle.c -- the CPU oracle for the W8A8 linear layer (test
 * infrastructure; see i8_oracle.h for the sources and the readings).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fopenmp -fPIC
 *        -shared.  No intrinsics, no BLAS, no reciprocal tricks: every step is
 * the plain definition, in the order the pages state it.
 *
 * Pins (tests/test_oracle.py checks each against something other than this
 * file):
 *   orc_f32_to_bf16    torch's fp32->bf16 cast on random and edge bit patterns
 *   orc_quant_rows     exact rational arithmetic (Python Fraction): the scale
 *                      is the fp32 nearest to absmax/127, every code is within
 *                      1/2 of x/scale, ties go to even, multiples j*scale give
 *                      code j, the zero row gives scale 0 and codes 0
 *   orc_gemm_s32       numpy int64 matmul; all-ones (acc = K), identity
 *                      weights, +-127 extremes at K = 131072
 *   orc_dequant_bias   fp64 evaluation rounded to bf16 (within 1 ulp), zero
 *                      accumulator gives the bias, unit scales give
 *                      bf16(acc + bias) exactly
 *
 * The pins are tested in turn: tests/test_oracle_mutants.py plants one
 * plausible mistake at a time in a copy of this file or of its wrapper (a
 * wrong constant, rounding mode, sign, index or operand order, a dropped
 * term) and requires each copy to fail at least one pin.
 */
#include "i8_oracle.h"

#include <math.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u) {
    /* NaN: keep the sign, force a quiet NaN payload. */
    return (uint16_t)((u >> 16) | 0x0040u);
  }
  /* Round to nearest even on the 16 bits that are dropped. */
  uint32_t lsb = (u >> 16) & 1u;
  uint32_t rounded = u + 0x7fffu + lsb;
  return (uint16_t)(rounded >> 16);
}

/* One row: absmax, scale = absmax / 127, q = clamp(rint(x / scale)). */
static void quant_one_row(const uint16_t* x, int64_t K, int8_t* q,
                          float* scale) {
  float amax = 0.0f;
  for (int64_t k = 0; k < K; ++k) {
    float v = fabsf(orc_bf16_to_f32(x[k]));
    if (v > amax) amax = v;
  }
  if (amax == 0.0f) {
    *scale = 0.0f;
    for (int64_t k = 0; k < K; ++k) q[k] = 0;
    return;
  }
  float s = amax / 127.0f; /* IEEE fp32 division, round to nearest even */
  *scale = s;
  for (int64_t k = 0; k < K; ++k) {
    float t = orc_bf16_to_f32(x[k]) / s; /* a true division, not x * (1/s) */
    float r = rintf(t);                   /* default mode: ties to even */
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[k] = (int8_t)r;
  }
}

int orc_quant_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                   int8_t* q, int64_t ldq, float* scale) {
  if (rows < 0 || K < 0 || ldx < K || ldq < K) return -1;
  if (rows > 0 && K > 0 && (!x || !q)) return -1;
  if (rows > 0 && !scale) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    quant_one_row(x + r * ldx, K, q + r * ldq, scale + r);
  }
  return 0;
}

int orc_gemm_s32(const int8_t* a, int64_t lda, const int8_t* w, int64_t ldw,
                 int64_t M, int64_t N, int64_t K, int32_t* c, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0 || K > 131072) return -1;
  if (lda < K || ldw < K || ldc < N) return -1;
  if (M > 0 && N > 0 && (!c || (K > 0 && (!a || !w)))) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    const int8_t* arow = a + m * lda;
    for (int64_t n = 0; n < N; ++n) {
      const int8_t* wrow = w + n * ldw;
      int32_t acc = 0;
      for (int64_t k = 0; k < K; ++k) {
        acc += (int32_t)arow[k] * (int32_t)wrow[k];
      }
      c[m * ldc + n] = acc;
    }
  }
  return 0;
}

int orc_dequant_bias(const int32_t* c, int64_t ldc, const float* s_a,
                     const float* s_w, const uint16_t* bias, int64_t M,
                     int64_t N, uint16_t* y, int64_t ldy) {
  if (M < 0 || N < 0 || ldc < N || ldy < N) return -1;
  if (M > 0 && N > 0 && (!c || !s_a || !s_w || !y)) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      float t = (float)c[m * ldc + n]; /* int32 -> fp32, nearest even */
      t = t * s_a[m];                  /* per-token scale */
      t = t * s_w[n];                  /* per-channel scale */
      t = t + (bias ? orc_bf16_to_f32(bias[n]) : 0.0f);
      y[m * ldy + n] = orc_f32_to_bf16(t);
    }
  }
  return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------ FP8
 * E4M3 as the OCP 8-bit floating point specification defines it: sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits.  Normal codes (exponent
 * field e = 1..15) hold (8 + m) * 2^(e - 10); subnormal codes (e = 0) hold
 * m * 2^-9; there is no infinity, and e = 15, m = 7 is NaN, so the largest
 * finite magnitude is 14 * 2^5 = 448.
 *
 * Pins (tests/test_oracle_fp8.py): torch's float8_e4m3fn cast on every bf16
 * value below the saturation point and on random fp32 patterns; the decode
 * of all 256 codes against the format's closed form; midpoints between
 * neighbouring codes (ties to the even code); the saturation rule; the
 * quantizer against exact rational arithmetic; the fp64 GEMM against
 * Python integer arithmetic on the codes scaled by 2^18; the epilogue against
 * its int32 counterpart on integer-valued accumulators. */

double orc_e4m3_to_f64(uint8_t b) {
  int e = (b >> 3) & 15;
  int m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return (b & 0x80) ? -v : v;
}

uint8_t orc_f32_to_e4m3(float f) {
  uint8_t sign;
  double a, quantum, r;
  int e2, lg, m;
  if (isnan(f)) return 0x7F;
  sign = signbit(f) ? 0x80 : 0x00;
  if (isinf(f)) return (uint8_t)(sign | 0x7E); /* saturate: +-448 */
  a = fabs((double)f);
  if (a == 0.0) return sign;
  /* The quantum of |f|'s binade: 2^(floor(log2 |f|) - 3) for normal
   * magnitudes, 2^-9 (the subnormal spacing) below 2^-6. */
  frexp(a, &e2);
  lg = e2 - 1;
  if (lg < -6) lg = -6;
  quantum = ldexp(1.0, lg - 3);
  /* a / quantum is exact (power-of-two divisor); nearbyint rounds half to
   * even, and an even multiple of the quantum is an even mantissa. */
  r = nearbyint(a / quantum) * quantum;
  if (r > 448.0) r = 448.0; /* finite saturation */
  if (r == 0.0) return sign;
  if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (int)(r / ldexp(1.0, -9)));
  frexp(r, &e2);
  lg = e2 - 1; /* r in [2^lg, 2^(lg+1)) */
  m = (int)(r / ldexp(1.0, lg - 3)) - 8;
  return (uint8_t)(sign | ((lg + 7) << 3) | m);
}

/* One row: absmax, scale = absmax / 448, q = E4M3(x / scale). */
static void quant_one_row_e4m3(const uint16_t* x, int64_t K, uint8_t* q,
                               float* scale) {
  float amax = 0.0f;
  for (int64_t k = 0; k < K; ++k) {
    float v = fabsf(orc_bf16_to_f32(x[k]));
    if (v > amax) amax = v;
  }
  if (amax == 0.0f) {
    *scale = 0.0f;
    for (int64_t k = 0; k < K; ++k) q[k] = 0;
    return;
  }
  float s = amax / 448.0f; /* IEEE fp32 division, round to nearest even */
  *scale = s;
  for (int64_t k = 0; k < K; ++k) {
    float t = orc_bf16_to_f32(x[k]) / s; /* a true fp32 division */
    q[k] = orc_f32_to_e4m3(t);
  }
}

int orc_quant_rows_e4m3(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                        uint8_t* q, int64_t ldq, float* scale) {
  if (rows < 0 || K < 0 || ldx < K || ldq < K) return -1;
  if (rows > 0 && K > 0 && (!x || !q)) return -1;
  if (rows > 0 && !scale) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    quant_one_row_e4m3(x + r * ldx, K, q + r * ldq, scale + r);
  }
  return 0;
}

int orc_gemm_e4m3_f64(const uint8_t* a, int64_t lda, const uint8_t* w, int64_t ldw,
                      int64_t M, int64_t N, int64_t K, int absval, double* c,
                      int64_t ldc) {
  double val[256];
  if (M < 0 || N < 0 || K < 0 || K > 131072) return -1;
  if (lda < K || ldw < K || ldc < N) return -1;
  if (M > 0 && N > 0 && (!c || (K > 0 && (!a || !w)))) return -1;
  for (int b = 0; b < 256; ++b) {
    double v = orc_e4m3_to_f64((uint8_t)b);
    val[b] = absval ? fabs(v) : v;
  }
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    const uint8_t* arow = a + m * lda;
    for (int64_t n = 0; n < N; ++n) {
      const uint8_t* wrow = w + n * ldw;
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        acc += val[arow[k]] * val[wrow[k]];
      }
      c[m * ldc + n] = acc;
    }
  }
  return 0;
}

int orc_dequant_bias_f64acc(const double* c, int64_t ldc, const float* s_a,
                            const float* s_w, const uint16_t* bias, int64_t M,
                            int64_t N, uint16_t* y, int64_t ldy) {
  if (M < 0 || N < 0 || ldc < N || ldy < N) return -1;
  if (M > 0 && N > 0 && (!c || !s_a || !s_w || !y)) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      float t = (float)c[m * ldc + n]; /* fp64 -> fp32, nearest even */
      t = t * s_a[m];
      t = t * s_w[n];
      t = t + (bias ? orc_bf16_to_f32(bias[n]) : 0.0f);
      y[m * ldy + n] = orc_f32_to_bf16(t);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------ fused
 * Pins (tests/test_oracle_fused.py): orc_f64_to_bf16 against exact rational
 * rounding; LayerNorm against torch's fp64 layer_norm, against closed forms
 * (symmetric rows, constant rows, power-of-two scaling) and its zero-mean /
 * unit-variance invariants; GELU against torch's fp64 gelu where that is
 * accurate (x > -8), against x * scipy's normal CDF below, and the identity
 * gelu(x) - gelu(-x) = x. */

uint16_t orc_f64_to_bf16(double v) {
  double a, q, r;
  int e2, lg;
  uint16_t sign;
  if (isnan(v)) return 0x7FC0;
  sign = signbit(v) ? 0x8000 : 0x0000;
  a = fabs(v);
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  if (a == 0.0) return sign;
  /* quantum of a's binade: 2^(floor(log2 a) - 7); subnormal spacing 2^-133 */
  frexp(a, &e2);
  lg = e2 - 1;
  if (lg < -126) lg = -126;
  q = ldexp(1.0, lg - 7);
  r = nearbyint(a / q) * q; /* a / q exact; ties to the even multiple */
  {
    float f = (float)r; /* r has at most 8 significant bits: exact in fp32 */
    uint32_t u;
    if (r > 3.3895313892515355e38) return (uint16_t)(sign | 0x7F80); /* overflow */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
  }
}

int orc_layernorm_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                       double eps, uint16_t* y, int64_t ldy) {
  if (rows < 0 || K <= 0 || ldx < K || ldy < K || !(eps >= 0.0)) return -1;
  if (rows > 0 && (!x || !y)) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * ldx;
    uint16_t* yr = y + r * ldy;
    double mu = 0.0, var = 0.0, rs;
    for (int64_t k = 0; k < K; ++k) mu += (double)orc_bf16_to_f32(xr[k]);
    mu /= (double)K;
    for (int64_t k = 0; k < K; ++k) {
      double d = (double)orc_bf16_to_f32(xr[k]) - mu;
      var += d * d;
    }
    var /= (double)K;
    rs = sqrt(var + eps);
    for (int64_t k = 0; k < K; ++k) {
      yr[k] = orc_f64_to_bf16(((double)orc_bf16_to_f32(xr[k]) - mu) / rs);
    }
  }
  return 0;
}

int orc_gelu_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                  uint16_t* y, int64_t ldy) {
  if (rows < 0 || K <= 0 || ldx < K || ldy < K) return -1;
  if (rows > 0 && (!x || !y)) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t k = 0; k < K; ++k) {
      /* GELU(v) = v * Phi(v), Phi the standard normal CDF.  Phi(v) is
       * (1 + erf(v / sqrt 2)) / 2 = erfc(-v / sqrt 2) / 2; the second form
       * has no cancellation for v < 0 (the first rounds to 0 below about
       * v = -8.3 even in fp64). */
      double v = (double)orc_bf16_to_f32(x[r * ldx + k]);
      double phi = v >= 0.0 ? 0.5 * (1.0 + erf(v / sqrt(2.0))) : 0.5 * erfc(-v / sqrt(2.0));
      y[r * ldy + k] = orc_f64_to_bf16(v * phi);
    }
  }
  return 0;
}
