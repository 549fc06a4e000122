// skinny.cuh -- the W8A8 GEMM for few tokens (M <= 16), weight streaming.
//
// Same operation as gemm.cuh (Fused INT8 GEMM Kernel for Ideogram 4.0, arXiv
// 2606.14598, abstract: int8 x int8 -> int32, per-token x per-channel dequant
// + bias -> bf16), for the skinny shapes where the weights dominate the bytes
// and the 128-row tensor-core tiles would be almost empty.
//
//   * grid = (ceil(N / 64), splits); a CTA owns 64 weight rows and a K range
//     of whole 512-wide chunks, streamed through a 2-stage TMA ring (128-byte
//     swizzle); the split count gives about two CTAs per SM.
//   * 4 warps x 16 weight rows; mma.sync m16n8k16 (fp16 in, fp32 out) with the
//     <= 16 token rows as the A operand and 8 weight rows as B.  Both operands
//     take the same permutation of K inside each 16-wide block (lane q of a
//     quad reads the 4 consecutive codes 4q..4q+3 as one word), which leaves
//     every dot product unchanged.
//   * fp32 partial sums are drained into int32 registers after every 512-K
//     chunk, so |partial| <= 127^2 * 512 < 2^24 stays exact in fp32.
//   * one K split: the CTA applies the epilogue itself; several: the int32
//     partials are added into an [M, N] buffer with integer atomics (exact,
//     order-independent) and the last CTA to finish an N-block (a counter per
//     block) applies the epilogue for that block.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "gemm.cuh"
#include "ptx.cuh"

namespace i8 {

struct SkinnyParams {
  int M, N, K;
  int num_kc;                 // K chunks of 512 in total
  int kc_per_cta;             // K chunks per split (grid.y splits)
  int out_mode;               // kOutBf16 or kOutInt32
  const int8_t* aq;           // [M, K]
  const float* s_a;
  const float* s_w;
  const uint16_t* bias;
  void* out;
  int64_t ldo;
  int32_t* acc;               // [M, N] int32, zeroed before the launch
  unsigned int* counters;     // [ceil(N / 64)], zeroed before the launch
};

// Zeroes the split-K workspace (n16 16-byte words) before the skinny kernel.
// A kernel rather than a memset so that it joins the stream's programmatic
// dependent launches: it waits for the previous kernel (which may still be
// reading this workspace) before writing, and lets the GEMM's prologue start
// early; the GEMM waits for it to finish before touching the workspace.
__global__ void __launch_bounds__(256) zero_ws_kernel(uint4* __restrict__ ws, int64_t n16) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    ws[i] = make_uint4(0u, 0u, 0u, 0u);
}

constexpr int kSkinnyRows = 64;
constexpr int kSkinnyK = 512;
constexpr int kCh = 4;   // independent accumulator chains per n8 group

template <bool W16>
struct SkinnyCfg {
  static constexpr int BOX_K = W16 ? 64 : 128;                    // elements per 128-byte row
  static constexpr int BOXES = kSkinnyK / BOX_K;                  // 4 (int8) or 8 (fp16)
  static constexpr int BOX_BYTES = kSkinnyRows * 128;             // 8 KB
  static constexpr int TILE_BYTES = BOXES * BOX_BYTES;            // 32 or 64 KB per stage
  static constexpr int STAGES = 2;
  static constexpr int SMEM_BYTES = STAGES * TILE_BYTES + 1024 + 64;
};

__device__ __forceinline__ void mma_m16n8k16_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool W16>
__global__ void __launch_bounds__(128) gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW,
                                                          const SkinnyParams p) {
  using Cfg = SkinnyCfg<W16>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);
  const uint32_t bar0 = sbase + Cfg::STAGES * Cfg::TILE_BYTES;
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem + Cfg::STAGES * Cfg::TILE_BYTES + 16);
  __shared__ int last_cta;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kSkinnyRows;
  const int kc0 = blockIdx.y * p.kc_per_cta;
  const int kc1 = min(kc0 + p.kc_per_cta, p.num_kc);
  const bool split = gridDim.y > 1;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  pdl_wait();  // weights, codes and the zeroed workspace may come from earlier work
  auto load_chunk = [&](int kc, int stage) {
    const uint32_t bar = bar0 + 8u * stage;
    mbar_arrive_expect_tx(bar, Cfg::TILE_BYTES);
    for (int b = 0; b < Cfg::BOXES; ++b)
      tma_load_2d(sbase + stage * Cfg::TILE_BYTES + b * Cfg::BOX_BYTES, &tmW, bar,
                  kc * kSkinnyK + b * Cfg::BOX_K, n0);
  };
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmW);
    load_chunk(kc0, 0);
    if (kc0 + 1 < kc1) load_chunk(kc0 + 1, 1);
  }

  const int g = lane >> 2;        // token row (and weight row within an n8 group)
  const int q = lane & 3;         // quad lane: codes 4q..4q+3 of each 16-block
  const int8_t* a_lo = p.aq + static_cast<int64_t>(g) * p.K;
  const int8_t* a_hi = p.aq + static_cast<int64_t>(g + 8) * p.K;
  const bool has_lo = g < p.M;
  const bool has_hi = g + 8 < p.M;

  int acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
  bool ok = true;
  uint32_t phase[2] = {0u, 0u};
  for (int kc = kc0; kc < kc1; ++kc) {
    const int stage = (kc - kc0) & 1;
    // this lane's token codes for the chunk, read while the tile lands
    uint32_t alo[kSkinnyK / 16], ahi[kSkinnyK / 16];
#pragma unroll
    for (int kb = 0; kb < kSkinnyK / 16; ++kb) {
      const int k = kc * kSkinnyK + kb * 16 + 4 * q;
      alo[kb] = (has_lo && k < p.K) ? __ldg(reinterpret_cast<const unsigned int*>(a_lo + k)) : 0u;
      ahi[kb] = (has_hi && k < p.K) ? __ldg(reinterpret_cast<const unsigned int*>(a_hi + k)) : 0u;
    }
    // block-uniform decision: every warp leaves the loop together, so the
    // __syncthreads below can never wait for a warp that gave up
    ok = __syncthreads_and(mbar_wait(bar0 + 8u * stage, phase[stage], abort_flag) ? 1 : 0) != 0;
    if (!ok) break;
    phase[stage] ^= 1u;
    const uint32_t tile = sbase + stage * Cfg::TILE_BYTES;
    // kCh independent accumulator chains per n8 group (16-blocks kb with the
    // same kb % kCh share one), so consecutive MMAs do not wait for each
    // other's results; each chain's fp32 partial is an exact integer below
    // 127^2 * 512 < 2^24, and so is their sum.
    float d[2][kCh][4];
#pragma unroll
    for (int grp = 0; grp < 2; ++grp)
#pragma unroll
      for (int c = 0; c < kCh; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[grp][c][i] = 0.0f;
#pragma unroll
    for (int kb = 0; kb < kSkinnyK / 16; ++kb) {
      uint32_t a0, a1, a2, a3;
      s8x4_to_f16x4(alo[kb], a0, a2);
      s8x4_to_f16x4(ahi[kb], a1, a3);
#pragma unroll
      for (int grp = 0; grp < 2; ++grp) {
        const int r = warp * 16 + grp * 8 + g;      // weight row within the tile
        uint32_t b0, b1;
        if constexpr (W16) {
          // fp16 codes: 4 codes = 8 bytes at byte offset 2 * (16 kb + 4 q)
          const int kbyte = 2 * (kb * 16 + 4 * q);
          const uint32_t addr = tile + (kbyte >> 7) * Cfg::BOX_BYTES + r * 128 +
                                ((((kbyte >> 4) & 7) ^ (r & 7)) << 4) + (kbyte & 15);
          asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(b0), "=r"(b1) : "r"(addr));
        } else {
          const int kbyte = kb * 16 + 4 * q;
          const uint32_t addr = tile + (kbyte >> 7) * Cfg::BOX_BYTES + r * 128 +
                                ((((kbyte >> 4) & 7) ^ (r & 7)) << 4) + (kbyte & 15);
          uint32_t wb;
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wb) : "r"(addr));
          s8x4_to_f16x4(wb, b0, b1);
        }
        mma_m16n8k16_f16(d[grp][kb % kCh], a0, a1, a2, a3, b0, b1);
      }
    }
    // every thread is done reading this stage: refill it two chunks ahead
    __syncthreads();
    if (threadIdx.x == 0 && kc + 2 < kc1) load_chunk(kc + 2, stage);
#pragma unroll
    for (int grp = 0; grp < 2; ++grp)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float t = d[grp][0][i];
#pragma unroll
        for (int c = 1; c < kCh; ++c) t = __fadd_rn(t, d[grp][c][i]);   // exact (integers < 2^24)
        acc[grp][i] += f32_exact_int_to_s32(__float_as_uint(t));
      }
  }

  pdl_trigger();
  // D fragment: acc[grp][0..1] -> token g, weight rows 2q, 2q+1 of the n8
  // group; acc[grp][2..3] -> token g + 8.
  if (!split) {
    if (!ok) return;
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      const int nb = n0 + warp * 16 + grp * 8 + 2 * q;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = g + (i >= 2 ? 8 : 0);
        const int n = nb + (i & 1);
        if (m < p.M && n < p.N) {
          if (p.out_mode == kOutBf16) {
            const float b = p.bias ? __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16) : 0.0f;
            const __nv_bfloat16 y = __float2bfloat16_rn(dequant_one(acc[grp][i], p.s_a[m], p.s_w[n], b));
            static_cast<uint16_t*>(p.out)[static_cast<int64_t>(m) * p.ldo + n] =
                *reinterpret_cast<const uint16_t*>(&y);
          } else {
            static_cast<int32_t*>(p.out)[static_cast<int64_t>(m) * p.ldo + n] = acc[grp][i];
          }
        }
      }
    }
    return;
  }
  if (ok) {
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      const int nb = n0 + warp * 16 + grp * 8 + 2 * q;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = g + (i >= 2 ? 8 : 0);
        const int n = nb + (i & 1);
        if (m < p.M && n < p.N && acc[grp][i] != 0)
          atomicAdd(p.acc + static_cast<int64_t>(m) * p.N + n, acc[grp][i]);
      }
    }
  }
  // The last CTA of this N-block applies the epilogue.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int prev = atomicAdd(p.counters + blockIdx.x, 1u);
    last_cta = (prev == gridDim.y - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!last_cta) return;
  __threadfence();
  const int cols = min(kSkinnyRows, p.N - n0);
  for (int e = threadIdx.x; e < p.M * cols; e += blockDim.x) {
    const int m = e / cols;
    const int n = n0 + e % cols;
    const int v = __ldcg(p.acc + static_cast<int64_t>(m) * p.N + n);
    if (p.out_mode == kOutBf16) {
      const float b = p.bias ? __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16) : 0.0f;
      const __nv_bfloat16 y = __float2bfloat16_rn(dequant_one(v, p.s_a[m], p.s_w[n], b));
      static_cast<uint16_t*>(p.out)[static_cast<int64_t>(m) * p.ldo + n] =
          *reinterpret_cast<const uint16_t*>(&y);
    } else {
      static_cast<int32_t*>(p.out)[static_cast<int64_t>(m) * p.ldo + n] = v;
    }
  }
}

}  // namespace i8
