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
//   * absmax on the raw bit patterns (|x| ordered like its bits), one
//     redux.sync per warp, shared memory across the G warps of a row;
//   * the quotient: t = x * fl(1/s) is within 2^-15 of the correctly rounded
//     fl(x / s) for every |x| <= amax when s is a normal float, so whenever t
//     is at least 2^-14 away from a half-integer both round to the same
//     integer; the rare near-tie elements (and rows with a subnormal scale)
//     take an IEEE division.  The result equals round_half_even(fl(x / s)).
//   * rounding to an integer uses the fp32 add of 1.5 * 2^23 (exact for
//     |t| <= 127.x, ties to even); the low byte of that sum's bit pattern is
//     the two's-complement int8 code.
#pragma once
#include <cstdint>

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

// One element: returns the fp32 bit pattern whose low byte is the code.
__device__ __forceinline__ uint32_t quant_one(float x, float s, float r, bool fast) {
  constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23
  constexpr float kNearTie = 0.5f - 0x1p-14f;
  float t = fminf(fmaxf(__fmul_rn(x, r), -127.0f), 127.0f);
  float y = __fadd_rn(t, kMagic);                // y - kMagic = round_half_even(t)
  float d = fabsf(__fadd_rn(t, -__fadd_rn(y, -kMagic)));
  if (!fast || d > kNearTie) {
    t = fminf(fmaxf(__fdiv_rn(x, s), -127.0f), 127.0f);
    y = __fadd_rn(t, kMagic);
  }
  return __float_as_uint(y);
}

// 8 bf16 (one 16-byte vector) -> 8 int8 codes packed in two words.
__device__ __forceinline__ uint2 quant_vec8(uint4 v, float s, float r, bool fast) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    b[2 * i] = quant_one(__uint_as_float(w[i] << 16), s, r, fast);
    b[2 * i + 1] = quant_one(__uint_as_float(w[i] & 0xFFFF0000u), s, r, fast);
  }
  // gather the low byte of each pattern: bytes {b0.0, b1.0, b2.0, b3.0}
  uint32_t lo = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
  uint32_t hi = __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410);
  return make_uint2(lo, hi);
}

// Grid: ceil(rows / (8 / G)) CTAs of 256 threads; warp w of a CTA serves row
// (blockIdx.x * (8 / G) + w / G), slice (w % G) of that row.
template <int V>
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t* __restrict__ x,
                                                         int64_t rows, int K, int64_t ldx,
                                                         int8_t* __restrict__ q, int64_t ldq,
                                                         float* __restrict__ scale, int G) {
  __shared__ uint32_t red[8];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rows_per_cta = 8 / G;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * rows_per_cta + warp / G;
  const int wig = warp % G;
  const bool valid_row = (warp / G) < rows_per_cta && row < rows;
  const int slice0 = wig * (32 * 8 * V);  // first element of this warp's slice

  const uint16_t* xr = x + (valid_row ? row : 0) * ldx;
  uint4 v[V];
  uint32_t amax2 = 0;  // two 15-bit |bf16| patterns, max taken lane-wise
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = slice0 + (i * 32 + lane) * 8;
    if (valid_row && e < K) {
      v[i] = ld_stream_v4(xr + e);
    } else {
      v[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) {
    amax2 = __vmaxu2(amax2, v[i].x & 0x7FFF7FFFu);
    amax2 = __vmaxu2(amax2, v[i].y & 0x7FFF7FFFu);
    amax2 = __vmaxu2(amax2, v[i].z & 0x7FFF7FFFu);
    amax2 = __vmaxu2(amax2, v[i].w & 0x7FFF7FFFu);
  }
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
  const float s = __fdiv_rn(amax, 127.0f);
  if (valid_row && wig == 0 && lane == 0) scale[row] = s;
  if (!valid_row) return;

  int8_t* qr = q + row * ldq;
  if (amax == 0.0f) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = slice0 + (i * 32 + lane) * 8;
      if (e < K) st_v2(qr + e, 0u, 0u);
    }
    return;
  }
  const bool fast = s >= 0x1p-126f;  // s normal: 1/s is finite and normal
  const float r = __frcp_rn(s);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = slice0 + (i * 32 + lane) * 8;
    if (e < K) {
      const uint2 c = quant_vec8(v[i], s, r, fast);
      st_v2(qr + e, c.x, c.y);
    }
  }
}

}  // namespace i8
