// gemm.cuh -- the fused W8A8 GEMM for sm_103a.
//
// Fused INT8 GEMM Kernel for Ideogram 4.0 (arXiv 2606.14598), abstract:
//   acc[m,n] = sum_k aq[m,k] * wq[n,k]          (int8 x int8 -> exact int32)
//   y[m,n]   = bf16(float(acc) * s_a[m] * s_w[n] + bias[n])   (epilogue)
//
// sm_103a has no INT8 tcgen05 MMA (the assembler rejects kind::i8 for this
// target).  The kernel therefore runs the int8 codes through the fp16 tensor
// pipe, exactly:
//   * every int8 code is exactly representable in fp16, every product
//     (|p| <= 127^2) is exact, and the fp32 accumulator is restarted every
//     `chunk` K-elements so that no partial sum reaches 2^24 (chunk <= 1024;
//     the default keeps partial sums below 2^23);
//   * each chunk's fp32 accumulator (integer-valued, hence exact) is read
//     from tensor memory, converted to int32 and summed in registers, so the
//     int32 result is exact for any K <= 131072.
//
// Structure (one persistent CTA per SM, warp-specialised):
//   warp 0        TMA producer: int8 A and B tiles (128-byte swizzle) into a
//                 ring of int8 stages; in the pre-widened-weights variant, B
//                 arrives as fp16 codes straight into the fp16 ring.
//   warp 1        TMEM allocator and single-thread tcgen05.mma issuer
//                 (M=128, N=BN, K=16 per instruction, fp32 accumulators).
//   warps 2-5     converters: int8 codes -> fp16 codes in the 128-byte-swizzled
//                 K-major layout the MMA descriptors expect.
//   warps 6-..    epilogue: drain chunk accumulators (two TMEM buffers, so the
//                 drain overlaps the next chunk's MMAs) into int32 registers,
//                 then dequantize + bias -> bf16, or store int32.
// Every pipeline wait is bounded (ptx.cuh); a timeout aborts the CTA cleanly.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace i8 {

enum GemmOut : int { kOutBf16 = 0, kOutInt32 = 1, kOutPartial = 2 };

struct GemmParams {
  int M, N, K;
  int num_m_blk, num_n_blk;
  int splits, kb_per_split, total_kb;  // K-blocks of 128
  int num_tiles;
  int chunk_stages;                    // fp16 stages (64 K each) per fp32 chunk
  int out_mode;                        // GemmOut
  const float* s_a;
  const float* s_w;
  const uint16_t* bias;                // may be null
  void* out;                           // y (bf16), c (int32) or workspace (int32)
  int64_t ldo;                         // elements
  int64_t split_stride;                // elements between split partials (kOutPartial)
};

template <int BN_, int S8_, int S16_, bool CONV_B_>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  static constexpr int S8 = S8_;
  static constexpr int S16 = S16_;
  static constexpr bool CONV_B = CONV_B_;
  static constexpr int BK8 = 128;   // int8 K per stage (one 128-byte row)
  static constexpr int BK16 = 64;   // fp16 K per stage (one 128-byte row)
  static constexpr int CONV_WARPS = 4;
  static constexpr int EPI_WARPS = BN / 32;  // 4 lane quarters x (BN / 128) column groups
  static constexpr int EPI_WARP0 = 2 + CONV_WARPS;
  static constexpr int NUM_WARPS = EPI_WARP0 + EPI_WARPS;
  static constexpr int THREADS = NUM_WARPS * 32;
  static constexpr int A8_BYTES = BM * BK8;
  static constexpr int B8_BYTES = CONV_B ? BN * BK8 : 0;
  static constexpr int A16_BYTES = BM * BK16 * 2;
  static constexpr int B16_BYTES = BN * BK16 * 2;
  static constexpr int OFF_A8 = 0;
  static constexpr int OFF_B8 = OFF_A8 + S8 * A8_BYTES;
  static constexpr int OFF_A16 = OFF_B8 + S8 * B8_BYTES;
  static constexpr int OFF_B16 = OFF_A16 + S16 * A16_BYTES;
  static constexpr int OFF_BAR = OFF_B16 + S16 * B16_BYTES;
  // full8[S8] empty8[S8] full16[S16] empty16[S16] accfull[2] accempty[2] done
  static constexpr int NUM_BARS = 2 * S8 + 2 * S16 + 5;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
  static constexpr int TMEM_COLS = 2 * BN;
  static_assert(BN == 128 || BN == 256, "BN");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void advance(int n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};

struct TileCoord {
  int mb, nb, ks, kb0, kb1;
};

__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, int tile) {
  TileCoord t;
  t.ks = tile % p.splits;
  const int rest = tile / p.splits;
  t.mb = rest % p.num_m_blk;
  t.nb = rest / p.num_m_blk;
  t.kb0 = t.ks * p.kb_per_split;
  t.kb1 = min(t.kb0 + p.kb_per_split, p.total_kb);
  return t;
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
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

// Convert the K-half `h` (int8 chunks 4h..4h+3) of row r of a swizzled int8
// tile into the fp16 tile of that half (chunks 0..7), both 128-byte rows with
// the 128-byte swizzle (16-byte chunk c of row r sits at c ^ (r & 7)).
__device__ __forceinline__ void convert_row_half(uint32_t src_tile, uint32_t dst_tile, int r,
                                                 int h) {
  const uint32_t srow = src_tile + static_cast<uint32_t>(r) * 128u;
  const uint32_t drow = dst_tile + static_cast<uint32_t>(r) * 128u;
  const int x = r & 7;
#pragma unroll
  for (int cl = 0; cl < 4; ++cl) {
    const uint4 v = lds128(srow + ((((h << 2) | cl) ^ x) << 4));
    uint4 o0, o1;
    s8x4_to_f16x4(v.x, o0.x, o0.y);
    s8x4_to_f16x4(v.y, o0.z, o0.w);
    s8x4_to_f16x4(v.z, o1.x, o1.y);
    s8x4_to_f16x4(v.w, o1.z, o1.w);
    sts128(drow + (((2 * cl) ^ x) << 4), o0);
    sts128(drow + (((2 * cl + 1) ^ x) << 4), o1);
  }
}

__device__ __forceinline__ int f32_exact_int_to_s32(uint32_t bits) {
  int v;
  asm("cvt.rni.s32.f32 %0, %1;" : "=r"(v) : "f"(__uint_as_float(bits)));
  return v;
}

__device__ __forceinline__ float dequant_one(int acc, float sa, float sw, float b) {
  float t = __int2float_rn(acc);
  t = __fmul_rn(t, sa);
  t = __fmul_rn(t, sw);
  return __fadd_rn(t, b);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Epilogue store of one thread's row segment (row m, 128 columns from n0).
template <int COLS>
__device__ __forceinline__ void store_row_segment(const GemmParams& p, int m, int n0,
                                                  const int (&acc)[COLS], int ks) {
  if (m >= p.M) return;
  if (p.out_mode == kOutBf16) {
    const float sa = p.s_a[m];
    uint16_t* yrow = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(m) * p.ldo;
#pragma unroll
    for (int j = 0; j < COLS; j += 8) {
      const int n = n0 + j;
      if (n >= p.N) break;
      if (n + 8 <= p.N) {
        const float4 w0 = *reinterpret_cast<const float4*>(p.s_w + n);
        const float4 w1 = *reinterpret_cast<const float4*>(p.s_w + n + 4);
        uint4 bb = make_uint4(0u, 0u, 0u, 0u);
        if (p.bias) bb = *reinterpret_cast<const uint4*>(p.bias + n);
        const float sw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float b0 = __uint_as_float(bw[i] << 16);
          const float b1 = __uint_as_float(bw[i] & 0xFFFF0000u);
          o[i] = pack_bf16x2(dequant_one(acc[j + 2 * i], sa, sw[2 * i], b0),
                             dequant_one(acc[j + 2 * i + 1], sa, sw[2 * i + 1], b1));
        }
        *reinterpret_cast<uint4*>(yrow + n) = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (n + i < p.N) {
            const float b = p.bias ? __uint_as_float(static_cast<uint32_t>(p.bias[n + i]) << 16) : 0.0f;
            const __nv_bfloat16 v = __float2bfloat16_rn(dequant_one(acc[j + i], sa, p.s_w[n + i], b));
            yrow[n + i] = *reinterpret_cast<const uint16_t*>(&v);
          }
        }
      }
    }
  } else {
    int32_t* crow = static_cast<int32_t*>(p.out) + static_cast<int64_t>(m) * p.ldo;
    if (p.out_mode == kOutPartial) crow += static_cast<int64_t>(ks) * p.split_stride;
#pragma unroll
    for (int j = 0; j < COLS; j += 4) {
      const int n = n0 + j;
      if (n >= p.N) break;
      if (n + 4 <= p.N) {
        *reinterpret_cast<int4*>(crow + n) = make_int4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n + i < p.N) crow[n + i] = acc[j + i];
      }
    }
  }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    gemm_w8a8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + Cfg::OFF_BAR;
  auto full8 = [&](int s) { return bar0 + 8u * s; };
  auto empty8 = [&](int s) { return bar0 + 8u * (Cfg::S8 + s); };
  auto full16 = [&](int s) { return bar0 + 8u * (2 * Cfg::S8 + s); };
  auto empty16 = [&](int s) { return bar0 + 8u * (2 * Cfg::S8 + Cfg::S16 + s); };
  auto accfull = [&](int b) { return bar0 + 8u * (2 * Cfg::S8 + 2 * Cfg::S16 + b); };
  auto accempty = [&](int b) { return bar0 + 8u * (2 * Cfg::S8 + 2 * Cfg::S16 + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * Cfg::S8 + 2 * Cfg::S16 + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::S8; ++s) {
      mbar_init(full8(s), 1);
      mbar_init(empty8(s), Cfg::CONV_WARPS);
    }
    for (int s = 0; s < Cfg::S16; ++s) {
      mbar_init(full16(s), Cfg::CONV_WARPS + (Cfg::CONV_B ? 0 : 1));
      mbar_init(empty16(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accfull(b), 1);
      mbar_init(accempty(b), Cfg::EPI_WARPS);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Ring r8, r16;
      for (int tile = blockIdx.x; tile < p.num_tiles && !*abort_flag; tile += gridDim.x) {
        const TileCoord tc = decode_tile(p, tile);
        for (int kb = tc.kb0; kb < tc.kb1; ++kb) {
          if (!mbar_wait(empty8(r8.s), r8.ph ^ 1u, abort_flag)) break;
          mbar_arrive_expect_tx(full8(r8.s), Cfg::A8_BYTES + Cfg::B8_BYTES);
          tma_load_2d(sbase + Cfg::OFF_A8 + r8.s * Cfg::A8_BYTES, &tmA, full8(r8.s), kb * Cfg::BK8,
                      tc.mb * Cfg::BM);
          if constexpr (Cfg::CONV_B) {
            tma_load_2d(sbase + Cfg::OFF_B8 + r8.s * Cfg::B8_BYTES, &tmB, full8(r8.s), kb * Cfg::BK8,
                        tc.nb * Cfg::BN);
          }
          r8.advance(Cfg::S8);
          if constexpr (!Cfg::CONV_B) {
            for (int h = 0; h < 2; ++h) {
              if (!mbar_wait(empty16(r16.s), r16.ph ^ 1u, abort_flag)) break;
              mbar_arrive_expect_tx(full16(r16.s), Cfg::B16_BYTES);
              tma_load_2d(sbase + Cfg::OFF_B16 + r16.s * Cfg::B16_BYTES, &tmB, full16(r16.s),
                          kb * Cfg::BK8 + h * Cfg::BK16, tc.nb * Cfg::BN);
              r16.advance(Cfg::S16);
            }
          }
          if (*abort_flag) break;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(Cfg::BM, Cfg::BN);
      Ring r16, racc;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const TileCoord tc = decode_tile(p, tile);
        const int nst = 2 * (tc.kb1 - tc.kb0);
        for (int st0 = 0; ok && st0 < nst; st0 += p.chunk_stages) {
          const int st1 = min(nst, st0 + p.chunk_stages);
          if (!(ok = mbar_wait(accempty(racc.s), racc.ph ^ 1u, abort_flag))) break;
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(racc.s * Cfg::BN);
          for (int st = st0; st < st1; ++st) {
            if (!(ok = mbar_wait(full16(r16.s), r16.ph, abort_flag))) break;
            tc_fence_after();
            const uint64_t ad = smem_desc_sw128(sbase + Cfg::OFF_A16 + r16.s * Cfg::A16_BYTES);
            const uint64_t bd = smem_desc_sw128(sbase + Cfg::OFF_B16 + r16.s * Cfg::B16_BYTES);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              mma_f16_ss(d, ad + 2u * j, bd + 2u * j, idesc, (st > st0 || j > 0) ? 1u : 0u);
            }
            mma_commit(empty16(r16.s));
            r16.advance(Cfg::S16);
          }
          if (!ok) break;
          mma_commit(accfull(racc.s));
          racc.advance(2);
        }
      }
      // Every MMA issued by this thread must finish before TMEM is released
      // (on the normal path they already have; after an abort some may not).
      mma_commit(done_bar);
      mbar_wait_bounded(done_bar, 0u, 100000000ull);
    }
  } else if (warp < Cfg::EPI_WARP0) {
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - 64;  // 0..127: the row this thread converts
    Ring r8, r16;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const TileCoord tc = decode_tile(p, tile);
      for (int kb = tc.kb0; kb < tc.kb1; ++kb) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(full8(r8.s), r8.ph, abort_flag));
        if (!ok) break;
        const uint32_t a8 = sbase + Cfg::OFF_A8 + r8.s * Cfg::A8_BYTES;
        const uint32_t b8 = sbase + Cfg::OFF_B8 + r8.s * Cfg::B8_BYTES;
        for (int h = 0; h < 2; ++h) {
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(empty16(r16.s), r16.ph ^ 1u, abort_flag));
          if (!ok) break;
          const uint32_t a16 = sbase + Cfg::OFF_A16 + r16.s * Cfg::A16_BYTES;
          convert_row_half(a8, a16, ct, h);
          if constexpr (Cfg::CONV_B) {
            const uint32_t b16 = sbase + Cfg::OFF_B16 + r16.s * Cfg::B16_BYTES;
#pragma unroll
            for (int r = ct; r < Cfg::BN; r += 128) convert_row_half(b8, b16, r, h);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full16(r16.s));
          r16.advance(Cfg::S16);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(empty8(r8.s));
        r8.advance(Cfg::S8);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - Cfg::EPI_WARP0;
    const int quarter = warp & 3;       // TMEM lanes this warp may access
    const int cg = ew >> 2;             // 128-column group
    Ring racc;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const TileCoord tc = decode_tile(p, tile);
      const int nst = 2 * (tc.kb1 - tc.kb0);
      int acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0;
      for (int st0 = 0; st0 < nst; st0 += p.chunk_stages) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(accfull(racc.s), racc.ph, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(racc.s * Cfg::BN + cg * 128);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(taddr + half * 64, r0);
          tmem_ld_32x32b_x32(taddr + half * 64 + 32, r1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            acc[half * 64 + i] += f32_exact_int_to_s32(r0[i]);
            acc[half * 64 + 32 + i] += f32_exact_int_to_s32(r1[i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accempty(racc.s));
        racc.advance(2);
      }
      if (!ok) break;
      const int m = tc.mb * Cfg::BM + quarter * 32 + lane;
      const int n0 = tc.nb * Cfg::BN + cg * 128;
      store_row_segment<128>(p, m, n0, acc, tc.ks);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// Split-K fix-up: exact int32 sum of the partials, then the same epilogue.
// One thread per 4 consecutive columns of one row.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const int32_t* __restrict__ ws,
                                                           int64_t split_stride, int64_t ldw,
                                                           int splits, GemmParams p) {
  const int groups_per_row = (p.N + 3) / 4;
  const int64_t total = static_cast<int64_t>(p.M) * groups_per_row;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(g / groups_per_row);
    const int n = static_cast<int>(g % groups_per_row) * 4;
    const int cnt = min(4, p.N - n);
    int acc[4] = {0, 0, 0, 0};
    const int32_t* src = ws + static_cast<int64_t>(m) * ldw + n;
    for (int s = 0; s < splits; ++s) {
      if (cnt == 4) {
        const int4 v = *reinterpret_cast<const int4*>(src + s * split_stride);
        acc[0] += v.x;
        acc[1] += v.y;
        acc[2] += v.z;
        acc[3] += v.w;
      } else {
        for (int i = 0; i < cnt; ++i) acc[i] += src[s * split_stride + i];
      }
    }
    if (p.out_mode == kOutBf16) {
      const float sa = p.s_a[m];
      uint16_t* yrow = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(m) * p.ldo;
      for (int i = 0; i < cnt; ++i) {
        const float b = p.bias ? __uint_as_float(static_cast<uint32_t>(p.bias[n + i]) << 16) : 0.0f;
        const __nv_bfloat16 v = __float2bfloat16_rn(dequant_one(acc[i], sa, p.s_w[n + i], b));
        yrow[n + i] = *reinterpret_cast<const uint16_t*>(&v);
      }
    } else {
      int32_t* crow = static_cast<int32_t*>(p.out) + static_cast<int64_t>(m) * p.ldo;
      for (int i = 0; i < cnt; ++i) crow[n + i] = acc[i];
    }
  }
}

}  // namespace i8
