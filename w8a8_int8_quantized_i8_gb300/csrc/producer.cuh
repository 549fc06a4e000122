// producer.cuh -- the per-token quantizer fused into the step that produces a
// linear layer's input.
//
// Fused INT8 GEMM Kernel for Ideogram 4.0 (arXiv 2606.14598): the fused GEMM
// saves the memory trip of the dequantize-to-bf16 path (aiexpert.news,
// mechanism paragraph).  The same argument applies one step earlier: in a DiT
// block every linear layer's input is produced by a LayerNorm (QKV,
// attention-out, MLP-up) or by the GELU (MLP-down), and quantizing that row in
// the producing kernel saves writing the bf16 row and reading it back.
//
// Definition (the oracle's): the producer's bf16 output y, then the per-row
// quantizer of y -- the codes are those the separate quantizer would give
// for the same bf16 row.
//   LayerNorm (no affine): mu = sum x / K, var = sum (x - mu)^2 / K,
//                          y = bf16((x - mu) * (1 / sqrt(var + eps)))
//   GELU (erf form):       y = bf16(0.5 x (1 + erf(x / sqrt 2))), evaluated as
//                          x * Phi(x) from one erfc(|x| / sqrt 2) (no cancellation)
// The reductions run in fp32 (per-lane, then warp shuffles, then across the
// row's warps), so y can differ from the oracle's fp64 value rounded once by
// one bf16 step where that value lies within fp32 noise of a rounding
// midpoint; the codes are then checked against the quantizer of the GPU's own
// y (an optional output), bit for bit.
//
// Layout and launch as quant_rows_kernel: one row per CTA, G warps per row,
// V 16-byte vectors per lane held in registers (K <= 8 * 32 * 16 * 8 = 32768).
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"
#include "quant.cuh"

namespace i8 {

enum ProducerOp : int { kOpLayerNorm = 0, kOpGelu = 1 };

// The two bf16 halves of a word as fp32 (exact widening).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two bf16 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&t);
}

// GELU in erf form, x * Phi(x) with Phi the standard normal CDF.  With
// t = erfc(|x| / sqrt 2): Phi(x) = 1 - t / 2 for x >= 0 and t / 2 for x < 0.
// One erfc per element, the same call on every lane (no divergent branch),
// and no cancellation: the naive 1 + erf(x / sqrt 2) is 6e-7 at x = -5,
// where fp32 resolves only 6e-8 near 1.
__device__ __forceinline__ float gelu_erf(float x) {
  constexpr float kRsqrt2 = 0.70710678118654752f;
  const float t = erfcf(fabsf(x) * kRsqrt2);
  const float phi = x >= 0.0f ? 1.0f - 0.5f * t : 0.5f * t;
  return x * phi;
}

// Sum over the CTA's G warps (every warp gets the total).  Each reduction
// of a row uses its own shared array, so one barrier per reduction suffices.
__device__ __forceinline__ float row_sum(float v, float* red, int warp, int lane, int G) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (G == 1) return v;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.0f;
  for (int j = 0; j < G; ++j) t += red[j];
  return t;
}

template <int V, int FMT, int OP>
__global__ void __launch_bounds__(256) producer_quant_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int K, int64_t ldx, float eps,
    int8_t* __restrict__ q, int64_t ldq, float* __restrict__ scale, uint16_t* __restrict__ y_out,
    int64_t ldy, int G) {
  __shared__ float red_a[8];
  __shared__ float red_b[8];
  __shared__ uint32_t red_m[8];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  const int slice0 = warp * (32 * 8 * V);
  const uint16_t* xr = x + row * ldx;
  // this warp's slice on its way into L2 while the previous kernel drains
  if (lane == 0 && slice0 < K)
    bulk_prefetch_l2(xr + slice0, static_cast<uint32_t>(min(32 * 8 * V, K - slice0)) * 2u);

  pdl_wait();  // X may be the previous kernel's output
  uint4 v[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = slice0 + (i * 32 + lane) * 8;
    v[i] = e < K ? ld_stream_v4(xr + e) : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_trigger();

  // ---- the producer: v (bf16 x) -> v (bf16 y), in registers
  if constexpr (OP == kOpLayerNorm) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) s += bf16_lo(w[j]) + bf16_hi(w[j]);   // padding adds 0
    }
    const float mean = __fdiv_rn(row_sum(s, red_a, warp, lane, G), static_cast<float>(K));
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = slice0 + (i * 32 + lane) * 8;
      if (e < K) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float d0 = bf16_lo(w[j]) - mean;
          const float d1 = bf16_hi(w[j]) - mean;
          ss += d0 * d0 + d1 * d1;
        }
      }
    }
    const float var = __fdiv_rn(row_sum(ss, red_b, warp, lane, G), static_cast<float>(K));
    const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
#pragma unroll
    for (int i = 0; i < V; ++i) {
      uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        w[j] = pack_bf16x2_rn(__fmul_rn(__fsub_rn(bf16_lo(w[j]), mean), rstd),
                              __fmul_rn(__fsub_rn(bf16_hi(w[j]), mean), rstd));
      }
      v[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = pack_bf16x2_rn(gelu_erf(bf16_lo(w[j])), gelu_erf(bf16_hi(w[j])));
      v[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }

  // ---- the per-row quantizer of y (same steps as quant_rows_kernel)
  uint32_t amax2 = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = slice0 + (i * 32 + lane) * 8;
    if (e < K) {
      amax2 = absmax_bf16x2(amax2, v[i].x);
      amax2 = absmax_bf16x2(amax2, v[i].y);
      amax2 = absmax_bf16x2(amax2, v[i].z);
      amax2 = absmax_bf16x2(amax2, v[i].w);
    }
  }
  amax2 &= 0x7FFF7FFFu;
  uint32_t abits = max(amax2 & 0xFFFFu, amax2 >> 16);
  abits = __reduce_max_sync(0xFFFFFFFFu, abits);
  if (G > 1) {
    if (lane == 0) red_m[warp] = abits;
    __syncthreads();
    abits = 0;
    for (int j = 0; j < G; ++j) abits = max(abits, red_m[j]);
  }
  const float amax = __uint_as_float(abits << 16);
  const float s = __fdiv_rn(amax, FMT == kQuantE4M3 ? 448.0f : 127.0f);
  if (warp == 0 && lane == 0) scale[row] = s;
  if (y_out) {
    uint16_t* yr = y_out + row * ldy;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = slice0 + (i * 32 + lane) * 8;
      if (e < K) *reinterpret_cast<uint4*>(yr + e) = v[i];
    }
  }
  int8_t* qr = q + row * ldq * (FMT == kQuantF16 ? 2 : 1);
  const bool fast = s >= 0x1p-126f;
  const float r = __frcp_rn(s);
  const unsigned long long rr = f2(r, r);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = slice0 + (i * 32 + lane) * 8;
    if (e < K) {
      uint2 c = make_uint2(0u, 0u);
      if (amax != 0.0f) {
        if constexpr (FMT == kQuantE4M3) c = quant_vec8_e4m3(v[i], s);
        else c = quant_vec8(v[i], s, rr, fast);
      }
      store_codes8<FMT>(qr, e, c);
    }
  }
}

// ----------------------------------------------------------------- GELU by table
// bf16 has 65536 bit patterns, so the correctly rounded GELU of every input
// fits a 128 KB table: g_gelu_table[b] = bf16_rne(x * Phi(x)) for x = the bf16
// with bits b, evaluated in fp64 (Phi(x) = erfc(-x / sqrt 2) / 2, no
// cancellation) and rounded once.  gelu_table_kernel fills it on the device,
// once per device; the GELU producer then streams rows through a copy of the
// table in shared memory.  The output is exactly the fp64 value rounded once,
// which is the oracle's definition.
static __device__ __align__(16) uint16_t g_gelu_table[65536];

__global__ void __launch_bounds__(256) gelu_table_kernel() {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= 65536) return;
  const double x = static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16));
  const double phi = 0.5 * erfc(-x * 0.70710678118654752440);
  const __nv_bfloat16 y = __double2bfloat16(x * phi);
  g_gelu_table[b] = *reinterpret_cast<const uint16_t*>(&y);
}

// Persistent: grid = SMs, 16 warps per CTA; the table is copied into shared
// memory once per CTA, then rows are processed R = 16 / G at a time (G warps
// per row, V 16-byte vectors per lane, as quant_rows_kernel).
template <int V, int FMT>
__global__ void __launch_bounds__(512, 1) gelu_table_quant_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int K, int64_t ldx, int8_t* __restrict__ q,
    int64_t ldq, float* __restrict__ scale, uint16_t* __restrict__ y_out, int64_t ldy, int G) {
  extern __shared__ __align__(16) uint16_t tab[];
  __shared__ uint32_t red_m[16];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int R = 16 / G;
  const int sub = warp / G;            // which row of the group of R
  const int wig = warp % G;
  const int slice0 = wig * (32 * 8 * V);
  {
    const uint4* src = reinterpret_cast<const uint4*>(g_gelu_table);
    uint4* dst = reinterpret_cast<uint4*>(tab);
    for (int i = threadIdx.x; i < 65536 / 8; i += 512) dst[i] = src[i];
  }
  __syncthreads();
  pdl_wait();  // X may be the previous kernel's output
  // One group of R rows at a time; the next group's loads are issued before
  // the current group is processed, so HBM stays busy during the table
  // lookups and reductions (one 512-thread CTA per SM holds few loads).
  auto load_rows = [&](int64_t b, uint4 (&dst)[V]) {
    const int64_t row = b + sub;
    const bool valid = row < rows;
    const uint16_t* xr = x + (valid ? row : 0) * ldx;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = slice0 + (i * 32 + lane) * 8;
      dst[i] = (valid && e < K) ? ld_stream_v4(xr + e) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // (rows of more than 8 vectors per lane keep a single buffer: two would
  // not fit the registers)
  constexpr bool kPrefetch = V <= 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * R;
  uint4 v[V], vn[kPrefetch ? V : 1];
  int64_t base = static_cast<int64_t>(blockIdx.x) * R;
  if (kPrefetch && base < rows) load_rows(base, v);
  for (; base < rows; base += stride) {
    if constexpr (kPrefetch) {
      if (base + stride < rows) load_rows(base + stride, vn);
    } else {
      load_rows(base, v);
    }
    const int64_t row = base + sub;
    const bool valid = row < rows;
    uint32_t amax2 = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = static_cast<uint32_t>(tab[w[j] & 0xFFFFu]) |
               (static_cast<uint32_t>(tab[w[j] >> 16]) << 16);
      v[i] = make_uint4(w[0], w[1], w[2], w[3]);
      const int e = slice0 + (i * 32 + lane) * 8;
      if (e < K) {
        amax2 = absmax_bf16x2(amax2, v[i].x);
        amax2 = absmax_bf16x2(amax2, v[i].y);
        amax2 = absmax_bf16x2(amax2, v[i].z);
        amax2 = absmax_bf16x2(amax2, v[i].w);
      }
    }
    amax2 &= 0x7FFF7FFFu;
    uint32_t abits = max(amax2 & 0xFFFFu, amax2 >> 16);
    abits = __reduce_max_sync(0xFFFFFFFFu, abits);
    if (G > 1) {
      if (lane == 0) red_m[warp] = abits;
      __syncthreads();
      abits = 0;
      for (int j = 0; j < G; ++j) abits = max(abits, red_m[sub * G + j]);
      __syncthreads();   // red_m is rewritten by the next group of rows
    }
    if (valid) {
      const float amax = __uint_as_float(abits << 16);
      const float s = __fdiv_rn(amax, FMT == kQuantE4M3 ? 448.0f : 127.0f);
      if (wig == 0 && lane == 0) scale[row] = s;
      if (y_out) {
        uint16_t* yr = y_out + row * ldy;
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const int e = slice0 + (i * 32 + lane) * 8;
          if (e < K) *reinterpret_cast<uint4*>(yr + e) = v[i];
        }
      }
      int8_t* qr = q + row * ldq * (FMT == kQuantF16 ? 2 : 1);
      const bool fast = s >= 0x1p-126f;
      const float r = __frcp_rn(s);
      const unsigned long long rr = f2(r, r);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = slice0 + (i * 32 + lane) * 8;
        if (e < K) {
          uint2 c = make_uint2(0u, 0u);
          if (amax != 0.0f) {
            if constexpr (FMT == kQuantE4M3) c = quant_vec8_e4m3(v[i], s);
            else c = quant_vec8(v[i], s, rr, fast);
          }
          store_codes8<FMT>(qr, e, c);
        }
      }
    }
    if constexpr (kPrefetch) {
#pragma unroll
      for (int i = 0; i < V; ++i) v[i] = vn[i];
    }
  }
  pdl_trigger();
}

}  // namespace i8
