/*
 * i8_oracle.h -- plain, slow, obviously-correct CPU definition of the W8A8
 * linear layer.  TEST INFRASTRUCTURE ONLY: only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this library.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * Sources (cited by title and passage; there are no numbered sections):
 *   [ABS]  "Realizing Native INT8 Compute for Diffusion Transformers on
 *          Consumer GPUs: A Fused INT8 GEMM Kernel for Ideogram 4.0"
 *          (arXiv 2606.14598), abstract -- the forward quantizes
 *          activations per token and weights per output channel, multiplies
 *          int8 by int8 into int32, and applies the per-token x per-channel
 *          dequantization and the bias in the GEMM epilogue, emitting bf16.
 *   [NEWS] aiexpert.news write-up of the same paper (Spanish), paragraph on
 *          the mechanism -- operands stay INT8, accumulation is int32, the
 *          epilogue dequantizes and adds the bias before writing bf16.
 *
 * Readings where the pages are silent (the plainest reading the rest supports):
 *   symmetric quantizer, no zero point; range +-127 (-128 never produced);
 *   scale = absmax / 127 in IEEE fp32; q = round-half-even(x / scale) with a
 *   true fp32 division; an all-zero row has scale 0 and codes 0; epilogue
 *   order float(acc) * s_a[m] * s_w[n] + bias[n], each step rounded to fp32
 *   (no FMA), then round-to-nearest-even to bf16; a missing bias adds +0.0f.
 *
 * bf16 values cross this interface as uint16_t bit patterns.
 * Parity status of each function: see the header comment in i8_oracle.c.
 */
#ifndef I8_ORACLE_H
#define I8_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* bf16 bit pattern -> fp32 (exact widening). */
float orc_bf16_to_f32(uint16_t b);
/* fp32 -> bf16 bit pattern, round to nearest, ties to even; NaN stays NaN. */
uint16_t orc_f32_to_bf16(float f);

/* Symmetric per-row INT8 quantizer ([ABS] per-token activations and
 * per-channel weights; both are "one scale per row of a K-contiguous
 * matrix").  x: rows x K bf16, row stride ldx elements.  q: rows x K int8,
 * row stride ldq.  scale: rows fp32.  Returns 0, or -1 on bad arguments. */
int orc_quant_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                   int8_t* q, int64_t ldq, float* scale);

/* acc[m][n] = sum_k a[m][k] * w[n][k] in int32 ([ABS] int8 x int8 -> int32).
 * a: M x K row-major (lda), w: N x K row-major (ldw, the [out,in] layout),
 * c: M x N row-major (ldc).  Requires K <= 131072 so that no int32 sum can
 * overflow (127*127*131072 < 2^31).  Returns 0, or -1 on bad arguments. */
int orc_gemm_s32(const int8_t* a, int64_t lda, const int8_t* w, int64_t ldw,
                 int64_t M, int64_t N, int64_t K, int32_t* c, int64_t ldc);

/* y[m][n] = bf16( ((float)acc[m][n] * s_a[m]) * s_w[n] + bias[n] )
 * ([ABS], [NEWS]: per-token x per-channel dequantization plus bias, bf16
 * out).  bias may be NULL (treated as +0.0f).  Returns 0, or -1. */
int orc_dequant_bias(const int32_t* c, int64_t ldc, const float* s_a,
                     const float* s_w, const uint16_t* bias, int64_t M,
                     int64_t N, uint16_t* y, int64_t ldy);

/* ------------------------------------------------------------------ FP8
 * The 8-bit floating-point arm: the pages set their INT8 kernel against an
 * FP8 baseline ([ABS]: the 172.9 s single-card FP8 run at 1024px, and the
 * closing remark that B200's native FP8 path beats the Ampere INT8 kernel).
 * They never print that quantizer.  Reading: the same
 * symmetric per-row scheme with the E4M3 format of the OCP 8-bit floating
 * point specification -- s = absmax / 448 in IEEE fp32 (448 = largest finite
 * E4M3 value), code = E4M3(fl32(x / s)) rounded to nearest, ties to even,
 * with finite saturation to +-448; the zero row gives s = 0 and codes 0.
 * E4M3 codes cross this interface as uint8_t bit patterns. */

/* fp32 -> E4M3 bit pattern: round to nearest even; finite values whose
 * rounded magnitude exceeds 448 saturate to +-448; NaN -> 0x7F. */
uint8_t orc_f32_to_e4m3(float f);
/* E4M3 bit pattern -> value (exact in fp64); the two NaN codes give NaN. */
double orc_e4m3_to_f64(uint8_t b);

/* Per-row E4M3 quantizer (same argument meaning as orc_quant_rows). */
int orc_quant_rows_e4m3(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                        uint8_t* q, int64_t ldq, float* scale);

/* c[m][n] = sum_k a[m][k] * w[n][k] over E4M3 codes, in fp64.  Exact for
 * K <= 131072: every product is an integer multiple of 2^-18 below 2^18, so
 * every partial sum is a multiple of 2^-18 below 2^35 and fits the 53-bit
 * significand.  absval != 0 sums |a * w| instead (used for error bounds).
 * Returns 0, or -1 on bad arguments. */
int orc_gemm_e4m3_f64(const uint8_t* a, int64_t lda, const uint8_t* w, int64_t ldw,
                      int64_t M, int64_t N, int64_t K, int absval, double* c,
                      int64_t ldc);

/* y[m][n] = bf16( ((float)c[m][n] * s_a[m]) * s_w[n] + bias[n] ): the same
 * epilogue steps as orc_dequant_bias, from an fp64 accumulator rounded once
 * to fp32 (nearest even).  bias may be NULL.  Returns 0, or -1. */
int orc_dequant_bias_f64acc(const double* c, int64_t ldc, const float* s_a,
                            const float* s_w, const uint16_t* bias, int64_t M,
                            int64_t N, uint16_t* y, int64_t ldy);

/* ------------------------------------------------------------------ fused
 * The step before the linear layer.  The pages' argument for folding the
 * dequantization into the GEMM epilogue is the memory trip it saves ([NEWS]
 * mechanism paragraph); the same argument moves the per-token quantizer into
 * the kernel that produces the layer's input: the LayerNorm in front of the
 * QKV, attention-out and MLP-up projections of a DiT block, and the GELU in
 * front of the MLP down-projection.  Definition: the producer's bf16 output,
 * then the per-row quantizer of that bf16 row -- so the fused path gives
 * exactly the codes of the unfused one whenever the bf16 rows agree. */

/* fp64 -> bf16 bit pattern with a single rounding (nearest, ties to even). */
uint16_t orc_f64_to_bf16(double v);

/* LayerNorm without affine parameters, per row, in fp64:
 *   mu = sum_k x_k / K,  var = sum_k (x_k - mu)^2 / K,
 *   y_k = bf16((x_k - mu) / sqrt(var + eps)), rounded once.
 * x, y: rows x K bf16 (row strides ldx, ldy).  Returns 0, or -1. */
int orc_layernorm_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                       double eps, uint16_t* y, int64_t ldy);

/* GELU (erf form) per element, in fp64:
 *   y = bf16(x * Phi(x)), Phi(x) = (1 + erf(x / sqrt 2)) / 2, evaluated as
 *   erfc(-x / sqrt 2) / 2 for x < 0; rounded once.  Returns 0, or -1. */
int orc_gelu_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                  uint16_t* y, int64_t ldy);

/* Threads the loops may use (OpenMP), or 1 when built without it. */
int orc_num_threads(void);
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
