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
