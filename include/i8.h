/*
 * i8.h -- C ABI of libi8, a GB300 (sm_103a) W8A8 INT8 linear layer.
 *
 * The operation is the one described in "Realizing Native INT8 Compute for
 * Diffusion Transformers on Consumer GPUs: A Fused INT8 GEMM Kernel for
 * Ideogram 4.0" (arXiv 2606.14598), abstract, and in the aiexpert.news
 * write-up of it (paragraph on the mechanism):
 *
 *   x  [M,K] bf16 activations  --per-token INT8 quant-->  aq [M,K] int8, s_a [M]
 *   w  [N,K] bf16 weights      --per-channel INT8 quant->  wq [N,K] int8, s_w [N]
 *   acc[m,n] = sum_k aq[m,k] * wq[n,k]                     (exact int32)
 *   y[m,n]   = bf16( float(acc) * s_a[m] * s_w[n] + bias[n] )   (epilogue)
 *
 * Quantizer (per row r of a K-contiguous matrix): amax = max_k |x[r,k]|,
 * scale = amax / 127 (IEEE fp32), q = clamp(round_half_even(x / scale),
 * -127, 127); an all-zero row gets scale 0 and codes 0.  The pages do not
 * print the quantizer; this symmetric form is the plain reading of their
 * scale-only epilogue.
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers of the current CUDA device, except
 *     where a call says otherwise.  The caller owns every buffer; the
 *     library allocates no device memory.  Work is queued on `stream`
 *     (NULL = legacy default stream) and the call returns without waiting.
 *   - Matrices are row-major with the contiguous dimension last; weights use
 *     the [out, in] = [N, K] layout, so both GEMM operands are K-contiguous.
 *   - bf16 buffers hold IEEE bfloat16 bit patterns (2 bytes per element).
 *   - Constraints: K % 16 == 0, 16 <= K <= 131072 (127*127*K must stay below
 *     2^31); M, N >= 0 and below 2^31; matrix base pointers 16-byte aligned;
 *     leading dimensions such that every row starts 16-byte aligned; scale
 *     pointer s_a 4-byte aligned; s_w and bias 16-byte aligned.
 *   - NaN or Inf inputs are outside the contract (results are unspecified,
 *     but no call faults on them).
 *   - Errors are returned, never thrown.  Argument, size and alignment errors
 *     are detected on the host before anything is queued.  Launch failures
 *     return I8_ERR_CUDA.  A kernel whose internal pipeline wait exceeds its
 *     time limit stops, records I8_ERR_DEVICE_TIMEOUT in a per-device status
 *     word and returns; i8_sync_check() reports (and clears) it.
 */
#ifndef I8_H
#define I8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle type (cudaStream_t), declared without
 * pulling in the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* i8_stream_t;

typedef enum {
  I8_OK = 0,
  I8_ERR_INVALID_ARG = 1,     /* NULL pointer, negative size, bad stride */
  I8_ERR_ALIGNMENT = 2,       /* pointer or row not 16-byte aligned */
  I8_ERR_UNSUPPORTED = 3,     /* K % 16 != 0, K > 131072, size out of range */
  I8_ERR_WORKSPACE = 4,       /* workspace missing or smaller than required */
  I8_ERR_CUDA = 5,            /* a CUDA runtime or launch error */
  I8_ERR_DEVICE_TIMEOUT = 6   /* a kernel's pipeline wait ran out of time */
} i8_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* i8_status_string(i8_status s);

/* Library version string, e.g. "i8 0.1.0 sm_103a". */
const char* i8_version(void);

/* Per-channel weight quantization (arXiv 2606.14598, abstract: weights are
 * quantized per output channel, offline, after training).
 *   w   [N,K] bf16, row stride ldw elements (ldw >= K, ldw % 8 == 0)
 *   wq  [N,K] int8, row stride ldq bytes (ldq >= K, ldq % 16 == 0)
 *   s_w [N]   fp32 per-channel scales                                     */
i8_status i8_quant_weight_perchannel(const void* w, int64_t N, int64_t K,
                                     int64_t ldw, int8_t* wq, int64_t ldq,
                                     float* s_w, i8_stream_t stream);

/* Per-token activation quantization (arXiv 2606.14598, abstract: one scale
 * per token; aiexpert.news mechanism paragraph: per-token activations).
 *   x   [M,K] bf16, row stride ldx elements (ldx >= K, ldx % 8 == 0)
 *   aq  [M,K] int8, row stride ldq bytes (ldq >= K, ldq % 16 == 0)
 *   s_a [M]   fp32 per-token scales                                       */
i8_status i8_quant_act_pertoken(const void* x, int64_t M, int64_t K,
                                int64_t ldx, int8_t* aq, int64_t ldq,
                                float* s_a, i8_stream_t stream);

/* Workspace bytes that i8_gemm_int32 / i8_gemm_dequant_bias_bf16 /
 * i8_gemm_dequant_bias_bf16_w16 need for this shape on the current device
 * (0 when the shape runs without a K split; the larger figure of the two
 * weight formats).  Returns 0 for shapes the GEMM rejects. */
size_t i8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Raw int32 accumulators, for checking (arXiv 2606.14598, abstract: the
 * int8 x int8 -> int32 accumulation is verified bit-exact against a library
 * integer GEMM).
 *   aq [M,K] int8 contiguous (row stride K), wq [N,K] int8 contiguous
 *   c  [M,N] int32, row stride ldc elements (ldc >= N, ldc % 4 == 0)
 *   ws / ws_bytes: device workspace of at least i8_gemm_workspace_bytes()
 *   (may be NULL when that is 0).  The result is exact whenever the true
 *   sum fits in int32: always for codes in -127..127, the quantizers' range
 *   (127 * 127 * 131072 < 2^31).  A -128 code is accepted too; the one sum
 *   that cannot be represented is +2^31, reached only when all 131072
 *   products of a row pair are (-128)^2, and that output is unspecified.  */
i8_status i8_gemm_int32(const int8_t* aq, const int8_t* wq, int64_t M,
                        int64_t N, int64_t K, int32_t* c, int64_t ldc,
                        void* ws, size_t ws_bytes, i8_stream_t stream);

/* The fused W8A8 GEMM (arXiv 2606.14598, abstract: int8 x int8 -> int32 with
 * the per-token x per-channel dequantization and the bias folded into the
 * epilogue; aiexpert.news mechanism paragraph: bf16 is emitted after the
 * epilogue).
 *   aq [M,K] int8 contiguous, s_a [M] fp32, wq [N,K] int8 contiguous,
 *   s_w [N] fp32, bias [N] bf16 or NULL (treated as +0),
 *   y  [M,N] bf16, row stride ldy elements (ldy >= N, ldy % 8 == 0)
 *   y[m,n] = bf16_rne(((float(acc) * s_a[m]) * s_w[n]) + bias[n]), each
 *   step an fp32 operation rounded to nearest even.                        */
i8_status i8_gemm_dequant_bias_bf16(const int8_t* aq, const float* s_a,
                                    const int8_t* wq, const float* s_w,
                                    const void* bias, int64_t M, int64_t N,
                                    int64_t K, void* y, int64_t ldy, void* ws,
                                    size_t ws_bytes, i8_stream_t stream);

/* ------------------------------------------------------------------ E4M3
 * The 8-bit floating-point arm (arXiv 2606.14598, abstract: the INT8 kernel
 * is set against an FP8 baseline, and the B200's native FP8 path beats it).
 * The pages print no FP8 quantizer; this library reads it as the same
 * symmetric per-row scheme with the E4M3 format of the OCP 8-bit floating
 * point specification (largest finite value 448):
 *   s = absmax / 448 (IEEE fp32), code = E4M3(fl32(x / s)) rounded to
 *   nearest even with finite saturation; the zero row gives s = 0, codes 0.
 * Codes are stored as their uint8_t bit patterns.  Same layouts, alignment
 * and error behaviour as the int8 quantizers above.                        */
i8_status i8_quant_weight_perchannel_e4m3(const void* w_bf16, int64_t N,
                                          int64_t K, int64_t ldw,
                                          uint8_t* wq, int64_t ldq,
                                          float* s_w, i8_stream_t stream);
i8_status i8_quant_act_pertoken_e4m3(const void* x_bf16, int64_t M,
                                     int64_t K, int64_t ldx, uint8_t* aq,
                                     int64_t ldq, float* s_a,
                                     i8_stream_t stream);

/* Workspace bytes the two E4M3 GEMM calls below need for this shape on the
 * current device: 0 when the shape runs without a K split, else the fp32
 * partials of the split (splits x M x round_up(N, 4) x 4 bytes).  Returns 0
 * for shapes the GEMM rejects. */
size_t i8_gemm_e4m3_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* fp32 accumulators of the E4M3 GEMM, for checking:
 *   c[m,n] = sum_k a[m,k] * w[n,k] over the decoded E4M3 codes, accumulated
 *   by the tensor core in fp32 (rounded; the order of its additions is not
 *   specified, so the result is within the fp32 accumulation bound of the
 *   exact sum, not bit-identical to a sequential loop).  When the shape's
 *   plan splits K, the splits' fp32 partials are added in split order (a
 *   fixed order: repeated calls give the same bits).
 *   aq [M,K], wq [N,K] E4M3 codes, contiguous (row stride K bytes)
 *   c  [M,N] fp32, row stride ldc elements (ldc >= N, ldc % 4 == 0)
 *   ws / ws_bytes: device workspace of at least
 *   i8_gemm_e4m3_workspace_bytes() (may be NULL when that is 0);
 *   I8_ERR_WORKSPACE when it is too small.
 *   K % 16 == 0, K <= 131072.                                              */
i8_status i8_gemm_e4m3_f32(const uint8_t* aq, const uint8_t* wq, int64_t M,
                           int64_t N, int64_t K, float* c, int64_t ldc,
                           void* ws, size_t ws_bytes, i8_stream_t stream);

/* The fused E4M3 GEMM: the fp32 accumulator above, then the same epilogue
 * as i8_gemm_dequant_bias_bf16:
 *   y[m,n] = bf16_rne(((acc * s_a[m]) * s_w[n]) + bias[n]), fp32 steps.
 *   aq [M,K] / wq [N,K] E4M3 codes contiguous, s_a [M] / s_w [N] fp32,
 *   bias [N] bf16 or NULL, y [M,N] bf16 (ldy >= N, ldy % 8 == 0);
 *   ws / ws_bytes as for i8_gemm_e4m3_f32.                                 */
i8_status i8_gemm_e4m3_dequant_bias_bf16(const uint8_t* aq, const float* s_a,
                                         const uint8_t* wq, const float* s_w,
                                         const void* bias, int64_t M,
                                         int64_t N, int64_t K, void* y,
                                         int64_t ldy, void* ws,
                                         size_t ws_bytes, i8_stream_t stream);

/* ------------------------------------------------------------------ fp16 codes
 * The exact W8A8 product with the int8 codes held in 16-bit containers: the
 * activation quantizer writes each int8 code as the fp16 value of the same
 * integer, and the weights are widened once offline (i8_widen_weight_codes).
 * The GEMM then feeds both operands to the tensor core's fp16 kind straight
 * from memory, with no on-chip widening; products are exact and the fp32
 * accumulator restarts every chunk (i8_set_option I8_OPT_CHUNK_K), so the
 * int32 result and the bf16 output are identical to the int8-code calls
 * above (arXiv 2606.14598, abstract: int8 x int8 -> int32, per-token x
 * per-channel dequantization and bias folded into the epilogue).  The codes
 * take twice the memory of int8 codes.
 *
 * i8_quant_act_pertoken_f16codes: the quantizer of i8_quant_act_pertoken;
 *   q16 [M,K] fp16 values (-127..127), row stride ldq elements
 *   (ldq >= K, ldq % 8 == 0).                                              */
i8_status i8_quant_act_pertoken_f16codes(const void* x_bf16, int64_t M,
                                         int64_t K, int64_t ldx, void* q16,
                                         int64_t ldq, float* s_a,
                                         i8_stream_t stream);

/* Workspace bytes of the two fp16-code GEMM calls below (0 when the shape
 * runs without a K split; else int32 partials, splits x M x round_up(N, 4)
 * x 4 bytes).  Returns 0 for shapes the GEMM rejects. */
size_t i8_gemm_f16codes_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Exact int32 accumulators from fp16 codes, for checking.
 *   a16 [M,K], w16 [N,K] fp16 code values, contiguous (row stride K)
 *   c [M,N] int32 (ldc >= N, ldc % 4 == 0); ws as above.                    */
i8_status i8_gemm_int32_f16codes(const void* a16, const void* w16, int64_t M,
                                 int64_t N, int64_t K, int32_t* c,
                                 int64_t ldc, void* ws, size_t ws_bytes,
                                 i8_stream_t stream);

/* The fused GEMM from fp16 codes: same result and epilogue as
 * i8_gemm_dequant_bias_bf16; y [M,N] bf16 (ldy >= N, ldy % 8 == 0). */
i8_status i8_gemm_dequant_bias_bf16_f16codes(const void* a16, const float* s_a,
                                             const void* w16,
                                             const float* s_w,
                                             const void* bias, int64_t M,
                                             int64_t N, int64_t K, void* y,
                                             int64_t ldy, void* ws,
                                             size_t ws_bytes,
                                             i8_stream_t stream);

/* ------------------------------------------------------------------ fused producers
 * The per-token quantizer fused into the kernel that produces a linear
 * layer's input (arXiv 2606.14598 folds the dequantization into the GEMM to
 * save a memory trip -- aiexpert.news mechanism paragraph; the same argument
 * applies to the step before the GEMM).  In a DiT block the QKV,
 * attention-out and MLP-up inputs are LayerNorm outputs and the MLP-down
 * input is a GELU output.
 *   result:  y = bf16(producer(x)) per row, then the per-row quantizer of y
 *            (int8 or E4M3 per fmt) -- the codes the separate quantizer gives
 *            for that bf16 row.
 *   LayerNorm: no affine parameters, mu and the biased variance over the row,
 *            y = bf16((x - mu) / sqrt(var + eps)); reductions in fp32, so y may
 *            differ from the exactly rounded value by one bf16 step where it
 *            lies within fp32 noise of a rounding midpoint.
 *   GELU:    erf form, y = bf16(0.5 x (1 + erf(x / sqrt 2))), fp32 arithmetic.
 *   x [M,K] bf16 (row stride ldx elements, ldx % 8 == 0), q [M,K] codes: int8
 *   or E4M3 bit patterns (row stride ldq bytes, ldq % 16 == 0), or, for
 *   I8_CODES_F16, the int8 codes as fp16 values (row stride ldq elements,
 *   ldq % 8 == 0); s_a [M] fp32;
 *   y [M,K] bf16 or NULL: when given, receives the bf16 producer output (for
 *   checking, or when the layer's input is also needed elsewhere).
 *   K % 16 == 0 and K <= 32768 (the row is held in registers); larger K is
 *   I8_ERR_UNSUPPORTED.  eps >= 0 and finite.  fmt: i8_code_format.        */
typedef enum { I8_CODES_INT8 = 0, I8_CODES_E4M3 = 1, I8_CODES_F16 = 2 } i8_code_format;
i8_status i8_layernorm_quant_act_pertoken(const void* x_bf16, int64_t M,
                                          int64_t K, int64_t ldx, float eps,
                                          int fmt, void* q, int64_t ldq,
                                          float* s_a, void* y_bf16,
                                          int64_t ldy, i8_stream_t stream);
i8_status i8_gelu_quant_act_pertoken(const void* x_bf16, int64_t M, int64_t K,
                                     int64_t ldx, int fmt, void* q,
                                     int64_t ldq, float* s_a, void* y_bf16,
                                     int64_t ldy, i8_stream_t stream);

/* i8_gemm_dequant_bias_bf16 for callers that cannot allocate device memory
 * at call time -- for example a plugin running inside another runtime that
 * offers no workspace hook, an application whose device memory is all owned
 * by a different allocator, or a latency-critical loop where cudaMalloc and
 * cudaFree (which may synchronize the device) are not allowed.  The paper has
 * no counterpart: this is a packaging variant of the fused GEMM.
 *   Same arguments and result as i8_gemm_dequant_bias_bf16, without ws and
 *   ws_bytes.  The split-K scratch lives in a fixed 16 MiB (16777216-byte)
 *   array inside the library, held on every GPU
 *   that loads the library until the process exits.  The launch plan is
 *   capped to that size: where the regular plan's scratch
 *   (i8_gemm_workspace_bytes) is larger, the call splits K fewer times, or
 *   not at all, and falls back from stream-K to whole tiles, with the same
 *   result bit for bit.  Only a plan that still needs more (a split count
 *   forced with I8_OPT_FORCE_SPLITS) is rejected with I8_ERR_WORKSPACE,
 *   before anything is queued.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture.  The call itself allocates nothing.
 *   All calls share the one array and it keeps the last call's contents.
 *   Split-K partials are written in full before they are read; the
 *   few-token kernel needs no scratch; stream-K arrival words carry a
 *   per-launch tag, so old words count as zero.  Calls whose
 *   kernels overlap on the GPU -- on different streams, or from different
 *   host threads -- race on the array; serialize them.                      */
i8_status i8_gemm_dequant_bias_bf16_noalloc(const int8_t* aq, const float* s_a,
                                            const int8_t* wq, const float* s_w,
                                            const void* bias, int64_t M,
                                            int64_t N, int64_t K, void* y,
                                            int64_t ldy, i8_stream_t stream);

/* Widens int8 weight codes to fp16 codes (the same integers, exactly), for
 * i8_gemm_dequant_bias_bf16_w16.  This is part of the offline weight
 * preparation, next to i8_quant_weight_perchannel: sm_103a has no INT8
 * tensor-core MMA, the GEMM runs the integer codes through the fp16 tensor
 * pipe, and a pre-widened weight copy saves the on-chip widening of the
 * weight operand on every call (at 2 bytes per weight in HBM).
 *   wq  [N,K] int8 contiguous;  w16 [N,K] fp16 bit patterns, contiguous.   */
i8_status i8_widen_weight_codes(const int8_t* wq, int64_t N, int64_t K,
                                void* w16, i8_stream_t stream);

/* i8_gemm_dequant_bias_bf16 with the weight codes given pre-widened to fp16
 * (from i8_widen_weight_codes).  Same arithmetic, bit-identical output.     */
i8_status i8_gemm_dequant_bias_bf16_w16(const int8_t* aq, const float* s_a,
                                        const void* w16, const float* s_w,
                                        const void* bias, int64_t M, int64_t N,
                                        int64_t K, void* y, int64_t ldy,
                                        void* ws, size_t ws_bytes,
                                        i8_stream_t stream);

/* Process-wide tuning knobs (not thread-safe; set them before launching).
 *   I8_OPT_CHUNK_K      K-elements per exact fp32 accumulation chunk inside
 *                       the GEMM: a multiple of 64 in [64, 1024] (default
 *                       1024: partial sums stay below 127*127*1024 < 2^24).
 *   I8_OPT_FORCE_SPLITS K-splits to use for every shape, on every GEMM route
 *                       (int8, fp16-held and E4M3 codes; at most one split
 *                       per K block, and at most 8 on the few-token
 *                       kernel); 0 = the plan's own choice.
 *   I8_OPT_MAX_CTAS     cap on the persistent grid (0 = one CTA per SM).
 *   I8_OPT_TILE_N       GEMM tile width, 128 or 256 (0 = the table).
 *   I8_OPT_CTA_PAIR     GEMM on CTA pairs (256 x 256 tiles per cluster of 2):
 *                       0 = the table (default: pairs for int8 weights when
 *                       the 256 x 256 tiles fill every pair of SMs), 1 = never,
 *                       2 = whenever M, N >= 256.
 *   I8_OPT_SKINNY_MAX_M token counts M up to this value (0..16, default 16)
 *                       use the weight-streaming kernel for few tokens
 *                       (measured faster than the tiled kernels at every
 *                       M <= 16 of the DiT shapes).
 *   I8_OPT_QUANT_VPL    quantizer: most 16-byte vectors one lane holds
 *                       (1..16, default 6); more warps share a row above.
 *   I8_OPT_PDL          1 (default): launch the kernels with programmatic
 *                       stream serialization, so a kernel is scheduled while
 *                       the previous one drains (each waits for the previous
 *                       kernel's memory before touching global memory);
 *                       0: plain stream-ordered launches.
 *   I8_OPT_QUANT_ROWS   quantizer rows per CTA, 1..8 (0 = chosen by shape).
 *   I8_OPT_STREAM_K     stream-K schedule for the CTA-pair kernel (equal
 *                       (tile, K-block) shares per pair, tiles cut between
 *                       pairs finished from exact int32 partials; it needs
 *                       workspace; with 64 or more K blocks, whole waves of
 *                       tiles first and only the rest shared): 1 (default)
 *                       where the table predicts a gain (at least half a
 *                       wave of tiles and whole tiles filling under 93 % of
 *                       the last wave), 2 whenever whole tiles leave pairs
 *                       idle, 0 never.
 *   I8_OPT_NVTX         1: every call of this header opens an NVTX range
 *                       named after the call (visible in Nsight timelines;
 *                       free when no tool is attached); 0 (default): none.
 *   I8_OPT_PAIR_STAGE_K K covered by one fp16 stage of the int8-code CTA-pair
 *                       GEMM, i.e. by one converter-to-MMA hand-off: 128
 *                       (two 64-K sub-tiles) or 64; 0 (default) = 128
 *                       whenever CHUNK_K is a multiple of 128, else 64.
 *   I8_OPT_RASTER       order of the output tiles in the tiled kernels: 1 M
 *                       blocks fastest, 2 N blocks fastest, 0 (default) N
 *                       fastest when M > N, else M fastest.  Results do not
 *                       depend on it.
 * Changing FORCE_SPLITS changes the *_workspace_bytes() results.
 *
 * The environment variable I8_OPTIONS, read once when the library is
 * loaded, sets options without code changes: a comma-separated list of
 * name=value pairs with the names chunk_k, force_splits, max_ctas, tile_n,
 * quant_vpl, cta_pair, skinny_max_m, pdl, quant_rows, stream_k, nvtx,
 * pair_stage_k, raster (for example "chunk_k=512,stream_k=0").  Entries with
 * an unknown name or an invalid value are ignored. */
typedef enum {
  I8_OPT_CHUNK_K = 1,
  I8_OPT_FORCE_SPLITS = 2,
  I8_OPT_MAX_CTAS = 3,
  I8_OPT_TILE_N = 4,
  I8_OPT_QUANT_VPL = 5,
  I8_OPT_CTA_PAIR = 6,
  I8_OPT_SKINNY_MAX_M = 7,
  I8_OPT_PDL = 8,
  I8_OPT_QUANT_ROWS = 9,
  I8_OPT_STREAM_K = 10,
  I8_OPT_NVTX = 11,
  I8_OPT_PAIR_STAGE_K = 12,
  I8_OPT_RASTER = 13
} i8_option;
i8_status i8_set_option(i8_option opt, int64_t value);
/* Current value of an option (I8_ERR_INVALID_ARG for an unknown option or a
 * NULL value pointer). */
i8_status i8_get_option(i8_option opt, int64_t* value);

/* The launch plan a GEMM entry point would choose for a shape: the library's
 * fixed shape -> configuration table, which stands where the pages' Triton
 * kernel autotunes per shape (arXiv 2606.14598, abstract: an autotuned
 * Triton kernel).  Nothing is launched and no memory is touched.
 *   route   the entry points the plan is for (i8_route).
 *   sms     > 0: describe the machine by hand, and the call needs no GPU:
 *           `pairs` = CTA pairs of the route's pair kernel resident at once
 *           (0 = sms / 2), `skinny_slots` = weight-streaming CTAs resident
 *           at once (0 = 2 * sms; clusters of K splits are assumed to pack
 *           those slots fully).  0: use the current device's own figures,
 *           including how many clusters of each size fit at once (needs the
 *           device; pairs and skinny_slots are then ignored).
 *   ws_cap  workspace bytes the plan may use (0 = unbounded; the no-alloc
 *           entry point plans with its fixed 16 MiB).
 *   out     host pointer, filled on I8_OK.
 * The options set with i8_set_option apply exactly as in the GEMM calls.
 * Errors: I8_ERR_INVALID_ARG (NULL out, M or N < 1, an unknown route, a
 * negative machine figure), I8_ERR_UNSUPPORTED (a K or size the GEMM
 * rejects), I8_ERR_CUDA (sms = 0 without a usable device). */
typedef enum {
  I8_ROUTE_INT8 = 0,      /* i8_gemm_int32, i8_gemm_dequant_bias_bf16(_noalloc) */
  I8_ROUTE_W16 = 1,       /* i8_gemm_dequant_bias_bf16_w16 */
  I8_ROUTE_F16CODES = 2,  /* i8_gemm_int32_f16codes, i8_gemm_dequant_bias_bf16_f16codes */
  I8_ROUTE_E4M3 = 3       /* i8_gemm_e4m3_f32, i8_gemm_e4m3_dequant_bias_bf16 */
} i8_route;

typedef enum {
  I8_KERNEL_SKINNY = 0,         /* weight-streaming kernel for a few tokens */
  I8_KERNEL_TILE = 1,           /* one CTA per 128 x tile_n output tile */
  I8_KERNEL_PAIR = 2,           /* CTA pairs, one 256 x 256 tile per pair */
  I8_KERNEL_PAIR_STREAM_K = 3,  /* the same with the stream-K schedule */
  I8_KERNEL_DIRECT = 4          /* CTA pairs fed fp16 or E4M3 codes by TMA */
} i8_kernel;

typedef struct {
  int32_t kernel;        /* i8_kernel */
  int32_t tile_m;        /* output rows of one work item (M for the skinny kernel) */
  int32_t tile_n;        /* output columns of one work item */
  int32_t num_m, num_n;  /* work items along M and along N */
  int32_t block_k;       /* K per K block (skinny kernel: per 256-K stage) */
  int32_t total_kb;      /* K blocks */
  int32_t splits;        /* K splits (1 = none; stream-K reports 1) */
  int32_t kb_per_split;  /* K blocks per split (the last may hold fewer) */
  int32_t grid;          /* CTAs of the GEMM launch */
  int32_t n_fastest;     /* tile order: 1 = N blocks fastest, 0 = M blocks */
  int64_t ws_bytes;      /* workspace the call needs (0 = none) */
  double model_us;       /* direct kernels: the split cost model's time (us,
                            up to a constant) for this plan; else 0 */
  int32_t sk_waves;      /* stream-K: whole waves of tiles before the split ones */
  int32_t sk_pairs;      /* stream-K: CTA pairs sharing the split tiles' units */
} i8_plan_info;

i8_status i8_plan_query(int64_t M, int64_t N, int64_t K, i8_route route, int sms,
                        int pairs, int skinny_slots, size_t ws_cap, i8_plan_info* out);

/* Failure-detection self-test: queues a one-thread kernel that waits on a
 * pipeline barrier nothing will ever complete, through the same bounded wait
 * the GEMM uses, with a limit of limit_ms (1..5000).  The wait runs out, the
 * kernel records I8_ERR_DEVICE_TIMEOUT in the device status word and returns
 * normally; the next i8_sync_check() reports it.  The GPU context stays
 * usable.  (No counterpart on the pages: this is the library's own check of
 * its timeout path.) */
i8_status i8_selftest_timeout(int limit_ms, i8_stream_t stream);

/* Waits for `stream`, then reads and clears the current device's status
 * word: I8_ERR_DEVICE_TIMEOUT if any kernel of this library timed out since
 * the last check, I8_ERR_CUDA on a CUDA error, else I8_OK. */
i8_status i8_sync_check(i8_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* I8_H */
