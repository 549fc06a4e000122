// quant.cuh -- symmetric per-row INT8 quantization (per-token activations,
// per-channel weights).
//
// Fused INT8 GEMM Kernel for Ideogram 4.0 (arXiv 2606.14598), abstract: the
// forward quantizes activations per token and weights per output channel.
// Both are "one scale per row of a K-contiguous bf16 matrix":
//   amax = max_k |x[k]|,  s = amax / 127 (IEEE fp32),
//   q[k] = clamp(round_half_even(x[k] / s), -127, 127),  amax == 0 -> s = 0, q = 0.
//
// Design (HBM-bound: 2 bytes read + 1 byte written per element):
//   * a group of G warps owns one row; every lane holds V 16-byte vectors
//     (8 bf16 each) of the row in registers, so X is read from HBM once;
//   * absmax per lane with the packed bf16x2 |max| (exact: it returns one of
//     its inputs), one redux.sync per warp, shared memory across the G warps
//     of a row;
//   * the quotient: t = x * fl(1/s) is within 2^-15 of the correctly rounded
//     fl(x / s) for every |x| <= amax when s is a normal float, so whenever t
//     is at least 2^-14 away from a half-integer both round to the same
//     integer; a vector of 8 with any near-tie element (and every row with a
//     subnormal scale) takes an IEEE division instead.  The result equals
//     round_half_even(fl(x / s)); the clamp to +-127 can only bind on that
//     slow path (|t| <= 127 * (1 + 2^-22) when s is normal).
//   * fp32 pairs run through the packed f32x2 instructions.
//   * rounding to an integer uses the fp32 add of 1.5 * 2^23 (exact for
//     |t| <= 127.x, ties to even); the low byte of that sum's bit pattern is
//     the two's-complement int8 code.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace i8 {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// Packed fp32 pairs (f32x2 arithmetic, IEEE round-to-nearest per lane).
__device__ __forceinline__ unsigned long long f2(float lo, float hi) {
  unsigned long long d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_split(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Low bytes of four fp32 bit patterns -> one word (first pattern in byte 0).
__device__ __forceinline__ uint32_t low_bytes4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

constexpr float kRoundMagic = 12582912.0f;     // 1.5 * 2^23: adding it rounds to an integer
constexpr float kNearTie = 0.5f - 0x1p-14f;

// Exact path for one element: clamp(x / s) rounded half-to-even, as the
// bit pattern of (q + 1.5 * 2^23) whose low byte is the code.
__device__ __forceinline__ uint32_t quant_exact(float x, float s) {
  const float t = fminf(fmaxf(__fdiv_rn(x, s), -127.0f), 127.0f);
  return __float_as_uint(__fadd_rn(t, kRoundMagic));
}

// 8 bf16 (one 16-byte vector) -> 8 int8 codes packed in two words.
__device__ __forceinline__ uint2 quant_vec8(uint4 v, float s, unsigned long long rr, bool fast) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const unsigned long long mm = f2(kRoundMagic, kRoundMagic);
  uint32_t b[8];
  float dmax = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const unsigned long long x = f2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    const unsigned long long t = f2_mul(x, rr);         // x * fl(1/s)
    // y rounds t to an integer (+ magic).  If the compiler fuses the
    // multiply into this add, y rounds the exact product x * fl(1/s)
    // instead; that is also within 3 * 127 * 2^-24 of x / s, so the near-tie
    // test below covers both forms.
    const unsigned long long y = f2_add(t, mm);
    const unsigned long long d = f2_sub(t, f2_sub(y, mm));  // t - rint(t), exact
    float y0, y1, d0, d1;
    f2_split(y, y0, y1);
    f2_split(d, d0, d1);
    b[2 * i] = __float_as_uint(y0);
    b[2 * i + 1] = __float_as_uint(y1);
    dmax = fmaxf(dmax, fmaxf(fabsf(d0), fabsf(d1)));
  }
  if (!fast || dmax > kNearTie) {
    // a near-tie somewhere in the vector (or a subnormal scale): IEEE division
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      b[2 * i] = quant_exact(__uint_as_float(w[i] << 16), s);
      b[2 * i + 1] = quant_exact(__uint_as_float(w[i] & 0xFFFF0000u), s);
    }
  }
  return make_uint2(low_bytes4(b[0], b[1], b[2], b[3]), low_bytes4(b[4], b[5], b[6], b[7]));
}

// Four int8 codes -> four fp16 values (exact).  x ^ 0x80 is x + 128 as an
// unsigned byte u; the fp16 bit pattern 0x64uu is 1024 + u; subtracting
// 1152 (0x6480) leaves x.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// Stores 8 codes at element e of a code row: one byte each, or, for the
// fp16-code format, the same integers as fp16 values (16 bytes).
template <int FMT>
__device__ __forceinline__ void store_codes8(int8_t* qrow, int e, uint2 c);

// Two fp32 values -> two E4M3 codes (lo in byte 0), round to nearest even,
// finite saturation to +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// 8 bf16 (one 16-byte vector) -> 8 E4M3 codes packed in two words, each
// from the correctly rounded fp32 quotient x / s.
__device__ __forceinline__ uint2 quant_vec8_e4m3(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    c[i] = e4m3x2(__fdiv_rn(__uint_as_float(w[i] << 16), s),
                  __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), s));
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// Lane-wise max of |a| and |b| over bf16 pairs; the result's sign bits are
// the xor of the inputs' signs and are masked off by the caller.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// kQuantF16: the int8 decision, each code stored as the fp16 value of the
// same integer (2 bytes per code), ready for the tensor core's fp16 kind.
enum QuantFmt : int { kQuantInt8 = 0, kQuantE4M3 = 1, kQuantF16 = 2 };

template <int FMT>
__device__ __forceinline__ void store_codes8(int8_t* qrow, int e, uint2 c) {
  if constexpr (FMT == kQuantF16) {
    uint4 o;
    s8x4_to_f16x4(c.x, o.x, o.y);
    s8x4_to_f16x4(c.y, o.z, o.w);
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(qrow + 2 * e), "r"(o.x),
                 "r"(o.y), "r"(o.z), "r"(o.w)
                 : "memory");
  } else {
    st_v2(qrow + e, c.x, c.y);
  }
}

// Grid: ceil(rows / R) CTAs of 32 * G * R threads (G * R <= 8); warp w of a
// CTA serves row (blockIdx.x * R + w / G), slice (w % G) of that row.
// FMT selects the code format: int8 or E4M3 (one byte per code), or fp16
// values of the int8 codes (two bytes; ldq then counts fp16 elements).
template <int V, int FMT = kQuantInt8>
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t* __restrict__ x,
                                                         int64_t rows, int K, int64_t ldx,
                                                         int8_t* __restrict__ q, int64_t ldq,
                                                         float* __restrict__ scale, int G) {
  __shared__ uint32_t red[8];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rows_per_cta = static_cast<int>(blockDim.x >> 5) / G;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * rows_per_cta + warp / G;
  const int wig = warp % G;
  const bool valid_row = (warp / G) < rows_per_cta && row < rows;
  const int slice0 = wig * (32 * 8 * V);  // first element of this warp's slice
  const uint16_t* xr = x + (valid_row ? row : 0) * ldx;
  // Start this warp's slice on its way into L2 while the previous kernel of
  // the stream drains (a prefetch cannot leave stale data; the loads below
  // still wait for it).
  if (valid_row && lane == 0 && slice0 < K)
    bulk_prefetch_l2(xr + slice0, static_cast<uint32_t>(min(32 * 8 * V, K - slice0)) * 2u);

  pdl_wait();  // X may be the previous kernel's output
  uint4 v[V];
  uint32_t amax2 = 0;  // bf16x2 running max of |x| (sign bits meaningless)
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = slice0 + (i * 32 + lane) * 8;
    if (valid_row && e < K) {
      v[i] = ld_stream_v4(xr + e);
    } else {
      v[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  pdl_trigger();
#pragma unroll
  for (int i = 0; i < V; ++i) {
    amax2 = absmax_bf16x2(amax2, v[i].x);
    amax2 = absmax_bf16x2(amax2, v[i].y);
    amax2 = absmax_bf16x2(amax2, v[i].z);
    amax2 = absmax_bf16x2(amax2, v[i].w);
  }
  amax2 &= 0x7FFF7FFFu;
  uint32_t abits = max(amax2 & 0xFFFFu, amax2 >> 16);
  abits = __reduce_max_sync(0xFFFFFFFFu, abits);
  if (G > 1) {
    if (lane == 0) red[warp] = abits;
    __syncthreads();
    const int g0 = (warp / G) * G;
    abits = 0;
    for (int j = 0; j < G; ++j) abits = max(abits, red[g0 + j]);
  }
  const float amax = __uint_as_float(abits << 16);
  const float s = __fdiv_rn(amax, FMT == kQuantE4M3 ? 448.0f : 127.0f);
  if (valid_row && wig == 0 && lane == 0) scale[row] = s;
  if (!valid_row) return;

  int8_t* qr = q + row * ldq * (FMT == kQuantF16 ? 2 : 1);
  if (amax == 0.0f) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = slice0 + (i * 32 + lane) * 8;
      if (e < K) store_codes8<FMT>(qr, e, make_uint2(0u, 0u));
    }
    return;
  }
  if constexpr (FMT == kQuantE4M3) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = slice0 + (i * 32 + lane) * 8;
      if (e < K) {
        const uint2 c = quant_vec8_e4m3(v[i], s);
        st_v2(qr + e, c.x, c.y);
      }
    }
    return;
  }
  const bool fast = s >= 0x1p-126f;  // s normal: 1/s is finite and normal
  const float r = __frcp_rn(s);
  const unsigned long long rr = f2(r, r);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = slice0 + (i * 32 + lane) * 8;
    if (e < K) {
      const uint2 c = quant_vec8(v[i], s, rr, fast);
      store_codes8<FMT>(qr, e, c);
    }
  }
}

}  // namespace i8

namespace i8 {

// Rows longer than the register-resident kernel covers (8 warps x 32 lanes x
// 16 vectors x 8 = 32768 elements): one CTA of 256 threads per row, two
// passes over the row -- absmax, then the codes -- with the second pass's
// loads served mostly by L2.  The per-vector arithmetic is the same as the
// resident kernel's, so the codes are the same.
template <int FMT = kQuantInt8>
__global__ void __launch_bounds__(256) quant_rows_long_kernel(const uint16_t* __restrict__ x,
                                                              int64_t rows, int K, int64_t ldx,
                                                              int8_t* __restrict__ q,
                                                              int64_t ldq,
                                                              float* __restrict__ scale) {
  __shared__ uint32_t red[8];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  pdl_wait();
  if (row >= rows) return;
  const uint16_t* xr = x + row * ldx;
  const int vecs = K / 8;
  uint32_t amax2 = 0;
  for (int i = threadIdx.x; i < vecs; i += 256) {
    const uint4 v = ld_stream_v4(xr + 8 * i);
    amax2 = absmax_bf16x2(amax2, v.x);
    amax2 = absmax_bf16x2(amax2, v.y);
    amax2 = absmax_bf16x2(amax2, v.z);
    amax2 = absmax_bf16x2(amax2, v.w);
  }
  amax2 &= 0x7FFF7FFFu;
  uint32_t abits = max(amax2 & 0xFFFFu, amax2 >> 16);
  abits = __reduce_max_sync(0xFFFFFFFFu, abits);
  if (lane == 0) red[warp] = abits;
  __syncthreads();
  abits = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) abits = max(abits, red[j]);
  const float amax = __uint_as_float(abits << 16);
  const float s = __fdiv_rn(amax, FMT == kQuantE4M3 ? 448.0f : 127.0f);
  if (threadIdx.x == 0) scale[row] = s;
  int8_t* qr = q + row * ldq * (FMT == kQuantF16 ? 2 : 1);
  const bool fast = s >= 0x1p-126f;
  const float r = __frcp_rn(s);
  const unsigned long long rr = f2(r, r);
  for (int i = threadIdx.x; i < vecs; i += 256) {
    uint2 c = make_uint2(0u, 0u);
    if (amax != 0.0f) {
      const uint4 v = *reinterpret_cast<const uint4*>(xr + 8 * i);
      if constexpr (FMT == kQuantE4M3) c = quant_vec8_e4m3(v, s);
      else c = quant_vec8(v, s, rr, fast);
    }
    store_codes8<FMT>(qr, 8 * i, c);
  }
  pdl_trigger();
}

}  // namespace i8
