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
//     `chunk` K-elements so that no partial sum reaches 2^24 (chunk <= 1024,
//     the default: |partial| <= 127^2 * 1024 = 16516096 < 2^24; the GPU
//     tests confirm bit-exact int32 at every chunk length on adversarial
//     +-127 operands, so the tensor pipe keeps 24-bit integers exact);
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
//   warps 2-7     converters: int8 codes -> fp16 codes in the 128-byte-swizzled
//                 K-major layout the MMA descriptors expect.
//   warps 8-..    epilogue: drain chunk accumulators (two TMEM buffers, so the
//                 drain overlaps the next chunk's MMAs) into int32 registers,
//                 then dequantize + bias -> bf16 (or int32) into a swizzled
//                 shared-memory staging buffer and a bulk tensor store.
// Every pipeline wait is bounded (ptx.cuh); a timeout aborts the CTA cleanly.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"
#include "quant.cuh"

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
  // Stream-K schedule (CTA-pair kernel only): first sk_waves whole waves of
  // tiles (tile = pair + wave * P), then pair q < Q = sk_pairs takes the
  // units [q*U/Q, (q+1)*U/Q) of the U = (num_tiles - sk_waves * P) *
  // total_kb (tile, K-block) units of the remaining tiles, so every pair
  // does about the same work whatever the tile count.  A tile cut between
  // pairs is finished from exact int32 partials by the pair holding its first
  // K blocks.
  int stream_k;                        // 0: tile-strided schedule
  int sk_waves;                        // whole waves before the split tiles
  int sk_pairs;                        // Q: pairs sharing the split tiles' units
  unsigned long long* sk_arrive;       // [num_tiles][2] arrival words: epoch << 16 | count
  const int32_t* sk_part;              // [P][256][256] int32 partial slots
  unsigned long long sk_epoch;         // this launch's tag, in [1, 2^48)
  int n_fastest;                       // tile order: 0 M blocks fastest, 1 N blocks fastest
};

// Block coordinates of output tile `tile` in the schedule's order.  M blocks
// fastest: workers running at the same time share weight columns; N blocks
// fastest: they share activation rows.  The host picks the order that keeps
// the larger operand's reused part in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int tile, int& mb, int& nb) {
  if (p.n_fastest) {
    nb = tile % p.num_n_blk;
    mb = tile / p.num_n_blk;
  } else {
    mb = tile % p.num_m_blk;
    nb = tile / p.num_m_blk;
  }
}

// Kernel configuration.  CONV_A / CONV_B: the operand arrives as int8 codes
// and is widened to fp16 on chip; otherwise it arrives as fp16 codes through
// TMA (weights pre-widened offline; fp16 A is used only for calibration).
// Warp roles are warpgroup-aligned so that register budgets can be moved
// between roles with setmaxnreg:
//   warpgroup 0: warp 0 TMA producer, warp 1 MMA issuer, warps 2-3 converters
//   warpgroup 1: converters
//   warpgroups 2..: epilogue (BN / 128 warpgroups; one per 128 columns)
template <int BN_, int S8_, int S16_, bool CONV_A_, bool CONV_B_>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  static constexpr int S8 = S8_;
  static constexpr int S16 = S16_;
  static constexpr bool CONV_A = CONV_A_;
  static constexpr bool CONV_B = CONV_B_;
  static constexpr bool ANY_CONV = CONV_A || CONV_B;
  static constexpr bool ANY_DIRECT = !CONV_A || !CONV_B;
  static constexpr int BK8 = 128;   // int8 K per K-block (one 128-byte row)
  static constexpr int BK16 = 64;   // fp16 K per stage (one 128-byte row)
  static constexpr int CONV_WARPS = 6;
  static constexpr int CONV_THREADS = CONV_WARPS * 32;
  static constexpr int EPI_WARPS = BN / 32;   // 4 lane quarters x (BN / 128)
  static constexpr int EPI_WARP0 = 8;
  static constexpr int NUM_WARPS = EPI_WARP0 + EPI_WARPS;
  static constexpr int THREADS = NUM_WARPS * 32;
  // registers per thread after setmaxnreg (launch: 65536 / THREADS)
  static constexpr int REG_LO = BN == 256 ? 80 : 96;
  static constexpr int REG_HI = BN == 256 ? 176 : 232;
  static_assert(2 * 128 * REG_LO + (EPI_WARPS / 4) * 128 * REG_HI <=
                    THREADS * ((65536 / THREADS) & ~7),
                "register split exceeds the launch allocation");
  // conversion work per fp16 stage: one item = one 16-byte int8 chunk
  static constexpr int A_ITEMS = CONV_A ? BM * 4 : 0;
  static constexpr int B_ITEMS = CONV_B ? BN * 4 : 0;
  static constexpr int ITEMS = A_ITEMS + B_ITEMS;
  static constexpr int IPT = (ITEMS + CONV_THREADS - 1) / CONV_THREADS;
  // shared memory
  static constexpr int A8_BYTES = CONV_A ? BM * BK8 : 0;
  static constexpr int B8_BYTES = CONV_B ? BN * BK8 : 0;
  static constexpr int STAGE8 = A8_BYTES + B8_BYTES;
  static constexpr int A16_BYTES = BM * BK16 * 2;
  static constexpr int B16_BYTES = BN * BK16 * 2;
  static constexpr int STAGE16 = A16_BYTES + B16_BYTES;
  static constexpr int OFF_S8 = 0;
  static constexpr int OFF_S16 = OFF_S8 + (ANY_CONV ? S8 : 0) * STAGE8;
  static constexpr int OFF_EPI = OFF_S16 + S16 * STAGE16;   // 4 KB store staging per epilogue warp
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * 4096;
  // full8[S8] empty8[S8] full16[S16] empty16[S16] accfull[2] accempty[2] done
  static constexpr int NUM_BARS = 2 * S8 + 2 * S16 + 5;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr uint32_t TX8 = STAGE8;
  static constexpr uint32_t TX16 = (CONV_A ? 0 : A16_BYTES) + (CONV_B ? 0 : B16_BYTES);
  static constexpr uint32_t FULL16_COUNT = (ANY_CONV ? CONV_WARPS : 0) + (ANY_DIRECT ? 1 : 0);
  static_assert(BN == 128 || BN == 256, "BN");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(STAGE8 % 1024 == 0 && STAGE16 % 1024 == 0, "stage alignment");
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
  tile_coords(p, rest, t.mb, t.nb);
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

// s8x4_to_f16x4 (four int8 codes -> four fp16 values) lives in quant.cuh.

// One conversion item = one 16-byte chunk (16 int8 codes) of one row of an
// int8 stage, widened into two 16-byte chunks (16 fp16 codes) of the fp16
// stage of the same K-half.  Both tiles use the 128-byte swizzle: 16-byte
// chunk c of row r sits at position c ^ (r & 7) of the row's 128 bytes.
// Offsets are relative to the stage bases; the K-half h (int8 chunks 4h..4h+3)
// only flips bit 6 of the source offset, since (4h + c) ^ x == (c ^ x) ^ 4h.
struct ConvItem {
  uint32_t src;   // offset in the int8 stage, K-half 0
  uint32_t dst;   // offset of the first fp16 chunk (the second is dst ^ 16)
};

template <class Cfg>
__device__ __forceinline__ ConvItem conv_item(int i) {
  ConvItem it;
  int region8, region16, rows, idx;
  if (i < Cfg::A_ITEMS) {
    region8 = 0;
    region16 = 0;
    rows = Cfg::BM;
    idx = i;
  } else {
    region8 = Cfg::A8_BYTES;
    region16 = Cfg::A16_BYTES;
    rows = Cfg::BN;
    idx = i - Cfg::A_ITEMS;
  }
  const int cl = idx / rows;
  const int r = idx % rows;
  const int x = r & 7;
  it.src = static_cast<uint32_t>(region8 + r * 128 + ((cl ^ x) << 4));
  it.dst = static_cast<uint32_t>(region16 + r * 128 + (((2 * cl) ^ x) << 4));
  return it;
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
// The same steps from an fp32 accumulator (the E4M3 arm).
__device__ __forceinline__ float dequant_one(float acc, float sa, float sw, float b) {
  float t = __fmul_rn(acc, sa);
  t = __fmul_rn(t, sw);
  return __fadd_rn(t, b);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Epilogue store of one warp's 32 rows x 128 columns through a 4 KB
// shared-memory staging buffer (32 rows x 128 bytes, 128-byte swizzle) and a
// bulk tensor store per 128-byte-wide column group: bf16 groups are 64
// columns, int32 groups 32.  Lane i holds row (m_base + i) in acc[0..127].
// The tensor store clips rows >= M and columns >= N, so ragged tiles need no
// masking.  tmY is 3-D {N, M, splits}; z selects the split-K partial.
template <int COLS, typename Acc = int>
__device__ __forceinline__ void store_warp_tile_bf16(const GemmParams& p, const CUtensorMap* tmY,
                                                     uint32_t stage, int lane, int m_base, int n0,
                                                     const Acc (&acc)[COLS]) {
  const uint32_t row = stage + static_cast<uint32_t>(lane) * 128u;
  const uint32_t x = static_cast<uint32_t>(lane & 7);
  const int m = m_base + lane;
  {
    const float sa = m < p.M ? p.s_a[m] : 0.0f;
#pragma unroll
    for (int g = 0; g < COLS / 64; ++g) {
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      const int nb = n0 + g * 64;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int n = nb + 8 * c;
        float sw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        uint4 bb = make_uint4(0u, 0u, 0u, 0u);
        if (n + 8 <= p.N) {
          const float4 w0 = *reinterpret_cast<const float4*>(p.s_w + n);
          const float4 w1 = *reinterpret_cast<const float4*>(p.s_w + n + 4);
          sw[0] = w0.x; sw[1] = w0.y; sw[2] = w0.z; sw[3] = w0.w;
          sw[4] = w1.x; sw[5] = w1.y; sw[6] = w1.z; sw[7] = w1.w;
          if (p.bias) bb = *reinterpret_cast<const uint4*>(p.bias + n);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (n + i < p.N) {
              sw[i] = p.s_w[n + i];
              if (p.bias) {
                const uint32_t hb = p.bias[n + i];
                if (i & 1) reinterpret_cast<uint32_t*>(&bb)[i >> 1] |= hb << 16;
                else reinterpret_cast<uint32_t*>(&bb)[i >> 1] |= hb;
              }
            }
          }
        }
        const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = g * 64 + 8 * c + 2 * i;
          // ((float(acc) * s_a) * s_w) + bias, each step rounded to fp32.
          // Scalar __fmul_rn / __fadd_rn are never contracted into an FMA;
          // packed f32x2 mul + add were (one bf16 ulp off where the product
          // and the bias nearly cancel).
          const float lo = dequant_one(acc[j], sa, sw[2 * i], __uint_as_float(bw[i] << 16));
          const float hi =
              dequant_one(acc[j + 1], sa, sw[2 * i + 1], __uint_as_float(bw[i] & 0xFFFF0000u));
          o[i] = pack_bf16x2(lo, hi);
        }
        sts128(row + ((static_cast<uint32_t>(c) ^ x) << 4), make_uint4(o[0], o[1], o[2], o[3]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(tmY, stage, nb, m_base, 0);
        bulk_commit_group();
      }
    }
  }
}

// The same store with the per-channel scales and the bias already staged in
// shared memory (fp32 scales at sw, bf16 bias patterns at bias, both for
// columns n0, n0 + 1, ...; zero past N) and the row's per-token scale sa
// already loaded, so no global load sits between the accumulator and the
// bulk store.  All lanes read the same scale words (one broadcast each).
// F32_BITS: acc holds fp32 bit patterns (the E4M3 arm's accumulators)
// instead of exact int32 sums.
template <int COLS, bool F32_BITS = false>
__device__ __forceinline__ void store_warp_tile_bf16_staged(const CUtensorMap* tmY, uint32_t stage,
                                                            int lane, int m_base, int n0,
                                                            const int (&acc)[COLS], float sa,
                                                            uint32_t sw, uint32_t bias) {
  const uint32_t row = stage + static_cast<uint32_t>(lane) * 128u;
  const uint32_t x = static_cast<uint32_t>(lane & 7);
#pragma unroll
  for (int g = 0; g < COLS / 64; ++g) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int j = g * 64 + 8 * c;
      const uint4 w0 = lds128(sw + 4u * static_cast<uint32_t>(j));
      const uint4 w1 = lds128(sw + 4u * static_cast<uint32_t>(j) + 16u);
      const uint4 bb = lds128(bias + 2u * static_cast<uint32_t>(j));
      const uint32_t swb[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // ((float(acc) * s_a) * s_w) + bias, each step rounded to fp32
        // (scalar __fmul_rn / __fadd_rn: never contracted into an FMA)
        float lo, hi;
        if constexpr (F32_BITS) {
          lo = dequant_one(__int_as_float(acc[j + 2 * i]), sa, __uint_as_float(swb[2 * i]),
                           __uint_as_float(bw[i] << 16));
          hi = dequant_one(__int_as_float(acc[j + 2 * i + 1]), sa, __uint_as_float(swb[2 * i + 1]),
                           __uint_as_float(bw[i] & 0xFFFF0000u));
        } else {
          lo = dequant_one(acc[j + 2 * i], sa, __uint_as_float(swb[2 * i]),
                           __uint_as_float(bw[i] << 16));
          hi = dequant_one(acc[j + 2 * i + 1], sa, __uint_as_float(swb[2 * i + 1]),
                           __uint_as_float(bw[i] & 0xFFFF0000u));
        }
        o[i] = pack_bf16x2(lo, hi);
      }
      sts128(row + ((static_cast<uint32_t>(c) ^ x) << 4), make_uint4(o[0], o[1], o[2], o[3]));
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmY, stage, n0 + g * 64, m_base, 0);
      bulk_commit_group();
    }
  }
}

// Stages the per-channel scales and bias of columns [n0, n0 + 32 * nwarps)
// in shared memory: lane `lane` of warp `w` loads column n0 + 32 w + lane
// (zeros past N and for a missing bias).
__device__ __forceinline__ void stage_channel_scales(const GemmParams& p, uint32_t sw, uint32_t bias,
                                                     int n0, int w, int lane) {
  const int c = 32 * w + lane;
  const int n = n0 + c;
  float s = 0.0f;
  uint32_t b = 0;
  if (n < p.N) {
    s = p.s_w[n];
    if (p.bias) b = p.bias[n];
  }
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(sw + 4u * static_cast<uint32_t>(c)), "f"(s) : "memory");
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(bias + 2u * static_cast<uint32_t>(c)),
               "h"(static_cast<unsigned short>(b))
               : "memory");
}

// int32 values (results or partials) through the same staging buffer in
// 32-column groups; z selects the plane of the 3-D map tm.
template <int COLS>
__device__ __forceinline__ void store_warp_tile_s32(const CUtensorMap* tm, uint32_t stage, int lane,
                                                    int m_base, int n0, const int (&acc)[COLS],
                                                    int z) {
  const uint32_t row = stage + static_cast<uint32_t>(lane) * 128u;
  const uint32_t x = static_cast<uint32_t>(lane & 7);
  {
#pragma unroll
    for (int g = 0; g < COLS / 32; ++g) {
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int j = g * 32 + 4 * c;
        sts128(row + ((static_cast<uint32_t>(c) ^ x) << 4),
               make_uint4(static_cast<uint32_t>(acc[j]), static_cast<uint32_t>(acc[j + 1]),
                          static_cast<uint32_t>(acc[j + 2]), static_cast<uint32_t>(acc[j + 3])));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(tm, stage, n0 + g * 32, m_base, z);
        bulk_commit_group();
      }
    }
  }
}

template <int COLS>
__device__ __forceinline__ void store_warp_tile(const GemmParams& p, const CUtensorMap* tmY,
                                                uint32_t stage, int lane, int m_base, int n0,
                                                const int (&acc)[COLS], int z) {
  if (p.out_mode == kOutBf16) store_warp_tile_bf16<COLS>(p, tmY, stage, lane, m_base, n0, acc);
  else store_warp_tile_s32<COLS>(tmY, stage, lane, m_base, n0, acc, z);
}

// Epilogue role: drains chunk accumulators into int32 registers, then writes
// the tile (bf16 with dequant + bias, int32, or a split-K partial).
template <class Cfg>
__device__ __forceinline__ void gemm_epilogue_role(const GemmParams& p, const CUtensorMap* tmY,
                                                   uint32_t sbase, uint32_t tmem_base, int warp,
                                                   int lane, volatile int* abort_flag, uint32_t bar0) {
  auto accfull = [&](int b) { return bar0 + 8u * (2 * Cfg::S8 + 2 * Cfg::S16 + b); };
  auto accempty = [&](int b) { return bar0 + 8u * (2 * Cfg::S8 + 2 * Cfg::S16 + 2 + b); };
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
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + q4 * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[q4 * 32 + i] += f32_exact_int_to_s32(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accempty(racc.s));
      racc.advance(2);
    }
    if (!ok) break;
    const uint32_t stage = sbase + Cfg::OFF_EPI + static_cast<uint32_t>(ew) * 4096u;
    store_warp_tile<128>(p, tmY, stage, lane, tc.mb * Cfg::BM + quarter * 32,
                         tc.nb * Cfg::BN + cg * 128, acc, tc.ks);
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    gemm_w8a8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
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
  auto stage8 = [&](int s) { return sbase + Cfg::OFF_S8 + static_cast<uint32_t>(s * Cfg::STAGE8); };
  auto stage16 = [&](int s) { return sbase + Cfg::OFF_S16 + static_cast<uint32_t>(s * Cfg::STAGE16); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::S8; ++s) {
      mbar_init(full8(s), 1);
      mbar_init(empty8(s), Cfg::CONV_WARPS);
    }
    for (int s = 0; s < Cfg::S16; ++s) {
      mbar_init(full16(s), Cfg::FULL16_COUNT);
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
    tma_prefetch_desc(&tmY);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // operands and outputs may belong to the previous kernel

  if (warp >= Cfg::EPI_WARP0) {
    regs_inc<Cfg::REG_HI>();
    gemm_epilogue_role<Cfg>(p, &tmY, sbase, tmem_base, warp, lane, abort_flag, bar0);
  } else if (warp == 0) {
    regs_dec<Cfg::REG_LO>();
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Ring r8, r16;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const TileCoord tc = decode_tile(p, tile);
        for (int kb = tc.kb0; ok && kb < tc.kb1; ++kb) {
          if constexpr (Cfg::ANY_CONV) {
            if (!(ok = mbar_wait(empty8(r8.s), r8.ph ^ 1u, abort_flag))) break;
            mbar_arrive_expect_tx(full8(r8.s), Cfg::TX8);
            if constexpr (Cfg::CONV_A)
              tma_load_2d(stage8(r8.s), &tmA, full8(r8.s), kb * Cfg::BK8, tc.mb * Cfg::BM);
            if constexpr (Cfg::CONV_B)
              tma_load_2d(stage8(r8.s) + Cfg::A8_BYTES, &tmB, full8(r8.s), kb * Cfg::BK8,
                          tc.nb * Cfg::BN);
            r8.advance(Cfg::S8);
          }
          if constexpr (Cfg::ANY_DIRECT) {
            for (int h = 0; h < 2; ++h) {
              if (!(ok = mbar_wait(empty16(r16.s), r16.ph ^ 1u, abort_flag))) break;
              mbar_arrive_expect_tx(full16(r16.s), Cfg::TX16);
              const int k16 = kb * Cfg::BK8 + h * Cfg::BK16;
              if constexpr (!Cfg::CONV_A)
                tma_load_2d(stage16(r16.s), &tmA, full16(r16.s), k16, tc.mb * Cfg::BM);
              if constexpr (!Cfg::CONV_B)
                tma_load_2d(stage16(r16.s) + Cfg::A16_BYTES, &tmB, full16(r16.s), k16,
                            tc.nb * Cfg::BN);
              r16.advance(Cfg::S16);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    regs_dec<Cfg::REG_LO>();
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
            const uint64_t ad = smem_desc_sw128(stage16(r16.s));
            const uint64_t bd = smem_desc_sw128(stage16(r16.s) + Cfg::A16_BYTES);
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
  } else {
    regs_dec<Cfg::REG_LO>();
    // ------------------------------------------------------------ converters
    if constexpr (Cfg::ANY_CONV) {
      const int ct = threadIdx.x - 64;  // 0 .. CONV_THREADS-1
      ConvItem items[Cfg::IPT];
#pragma unroll
      for (int j = 0; j < Cfg::IPT; ++j) {
        const int i = ct + j * Cfg::CONV_THREADS;
        items[j] = conv_item<Cfg>(i < Cfg::ITEMS ? i : 0);
      }
      Ring r8, r16;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const TileCoord tc = decode_tile(p, tile);
        for (int kb = tc.kb0; kb < tc.kb1; ++kb) {
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(full8(r8.s), r8.ph, abort_flag));
          if (!ok) break;
          const uint32_t s8 = stage8(r8.s);
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(empty16(r16.s), r16.ph ^ 1u, abort_flag));
            if (!ok) break;
            const uint32_t s16 = stage16(r16.s);
            const uint32_t hx = static_cast<uint32_t>(h) << 6;
            uint4 v[Cfg::IPT];
#pragma unroll
            for (int j = 0; j < Cfg::IPT; ++j) {
              if (ct + j * Cfg::CONV_THREADS < Cfg::ITEMS) v[j] = lds128(s8 + (items[j].src ^ hx));
            }
#pragma unroll
            for (int j = 0; j < Cfg::IPT; ++j) {
              if (ct + j * Cfg::CONV_THREADS < Cfg::ITEMS) {
                uint4 o0, o1;
                s8x4_to_f16x4(v[j].x, o0.x, o0.y);
                s8x4_to_f16x4(v[j].y, o0.z, o0.w);
                s8x4_to_f16x4(v[j].z, o1.x, o1.y);
                s8x4_to_f16x4(v[j].w, o1.z, o1.w);
                sts128(s16 + items[j].dst, o0);
                sts128(s16 + (items[j].dst ^ 16u), o1);
              }
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
    }
  }

  __syncwarp();
  pdl_trigger();
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
  pdl_wait();  // the partials come from the GEMM kernel just before
  pdl_trigger();
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
