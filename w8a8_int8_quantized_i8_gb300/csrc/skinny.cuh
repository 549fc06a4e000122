// skinny.cuh -- the W8A8 GEMM for few tokens (M <= 16), weight streaming.
//
// Same operation as gemm.cuh (Fused INT8 GEMM Kernel for Ideogram 4.0, arXiv
// 2606.14598, abstract: int8 x int8 -> int32, per-token x per-channel dequant
// + bias -> bf16), for the skinny shapes where the weights dominate the bytes
// and the 128-row tensor-core tiles would be almost empty.
//
//   * A CTA owns 64 weight rows (an N-block) and a range of whole 256-K
//     stages.  The S <= 8 CTAs that split one N-block's K form a thread-block
//     cluster; grid = N-blocks x S, cluster rank = K split.
//   * One producer warp streams the CTA's weight rows and the token codes of
//     every stage through a ring of STAGES stages by TMA (128-byte swizzle);
//     two CTAs fit on an SM (int8 weights).
//     The parts of a box outside the tensors (rows past N, tokens past M, K
//     past its end) arrive as zeros and add nothing.  The weights of the
//     first fill are prefetched into L2 before the wait for the previous
//     kernel, so their DRAM latency overlaps its tail.
//   * Eight compute warps: warp w takes weight rows 16 (w % 4) .. + 16 and
//     K-half w / 4 of every stage, and runs mma.sync m16n8k16 (fp16 in, fp32
//     out) with the 16 weight rows as the A operand and the tokens (8, or 16
//     in two groups) as B.  Both operands take the same permutation of K
//     inside each 16-wide block (lane q of a quad reads the 4 consecutive
//     codes 4q..4q+3 as one word), which leaves every dot product unchanged.
//   * Four independent fp32 accumulator chains per token group, so
//     consecutive MMAs do not wait for each other; every 4 stages they are
//     summed and drained into int32 registers.  A warp's MMA covers 16 K, so
//     |partial| <= 16 * 127^2 = 258064; a chain gathers at most 8 of them and
//     the four chains' sum stays below 32 * 258064 < 2^24: exact in fp32.
//   * The warps' int32 partials meet in shared memory (integer adds).  With
//     one split the CTA applies the epilogue.  With S, cluster rank r owns a
//     slice of about 1/S of the outputs: every other CTA of the cluster adds
//     its partials of that slice into r's (red.async, counted on r's
//     mbarrier), and r applies the epilogue once they are all in.  No global
//     workspace, no atomics in global memory, nothing to clear between
//     calls, and no CTA waits for another except for the partials it owns.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "gemm.cuh"
#include "ptx.cuh"

namespace i8 {

struct SkinnyParams {
  int M, N, K;
  int num_ks;                 // 256-K stages in total: ceil(K / 256)
  int ks_per_cta;             // stages per K split
  int splits;                 // K splits = CTAs per cluster (1..kSkinnyMaxSplits)
  int out_mode;               // kOutBf16 or kOutInt32
  const float* s_a;
  const float* s_w;
  const uint16_t* bias;
  void* out;
  int64_t ldo;
};

constexpr int kSkinnyRows = 64;       // weight rows per CTA
constexpr int kSkinnyK = 256;         // K per stage
constexpr int kSkinnyMaxSplits = 8;   // portable cluster size
constexpr int kSkinnyMinStages = 4;   // least stages per K split (1024 K)
constexpr int kCh = 4;                // independent accumulator chains per token group
constexpr int kDrainStages = 4;       // stages between drains into int32

template <bool W16, int MT>
struct SkinnyCfg {
  static constexpr int BOX_K = W16 ? 64 : 128;                  // weight codes per 128-byte row
  static constexpr int W_BOXES = kSkinnyK / BOX_K;              // 2 (int8) or 4 (fp16 codes)
  static constexpr int W_BOX_BYTES = kSkinnyRows * 128;         // 8 KB
  static constexpr int A_BOXES = kSkinnyK / 128;                // token codes are int8
  static constexpr int A_ROWS = 8 * MT;                         // token rows per box
  static constexpr int A_BOX_BYTES = A_ROWS * 128;
  static constexpr int STAGE_BYTES = W_BOXES * W_BOX_BYTES + A_BOXES * A_BOX_BYTES;
  static constexpr int STAGES = W16 ? 4 : (MT == 1 ? 6 : 5);
  static constexpr int COMPUTE_WARPS = 8;
  static constexpr int THREADS = 32 * (COMPUTE_WARPS + 1);    // + the producer warp
  static constexpr int OFF_PART = STAGES * STAGE_BYTES;        // int32 [A_ROWS][64], token-major
  static constexpr int OFF_BAR = OFF_PART + A_ROWS * kSkinnyRows * 4;   // full[STAGES] empty[STAGES]
  static constexpr int OFF_FLAG = OFF_BAR + 2 * STAGES * 8;
  // the epilogue's constants: channel scales and bias (as fp32) of the 64
  // rows, token scales of the A_ROWS tokens
  static constexpr int OFF_SCL = OFF_FLAG + 16;
  // the mbarrier counting the other CTAs' adds into the owned slice
  static constexpr int OFF_REDBAR = (OFF_SCL + (2 * kSkinnyRows + A_ROWS) * 4 + 7) / 8 * 8;
  static constexpr int SMEM_BYTES = OFF_REDBAR + 8 + 1024;   // + 1 KB alignment room
  // two CTAs per SM: 228 KB per SM, 1 KB of it reserved per CTA
  static_assert(W16 || 2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs must fit on an SM");
  static_assert(SMEM_BYTES <= 227 * 1024, "more shared memory than a CTA may hold");
  static_assert(STAGE_BYTES % 1024 == 0 && W_BOX_BYTES % 1024 == 0 && A_BOX_BYTES % 1024 == 0,
                "128-byte-swizzled boxes must start on 1 KB boundaries");
  static_assert((kDrainStages * kSkinnyK / 2 / 16) / kCh * 16 * 127 * 127 * kCh < (1 << 24),
                "fp32 chains must stay exact between drains");
};

__device__ __forceinline__ void mma_m16n8k16_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

template <bool W16, int MT>
__global__ void __launch_bounds__(SkinnyCfg<W16, MT>::THREADS)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                       const SkinnyParams p) {
  using Cfg = SkinnyCfg<W16, MT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);
  const uint32_t full0 = sbase + Cfg::OFF_BAR;
  const uint32_t empty0 = full0 + 8u * Cfg::STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_FLAG);
  int* part = reinterpret_cast<int*>(smem + Cfg::OFF_PART);
  float* scl_w = reinterpret_cast<float*>(smem + Cfg::OFF_SCL);   // [64]
  float* scl_b = scl_w + kSkinnyRows;                              // [64]
  float* scl_a = scl_b + kSkinnyRows;                              // [A_ROWS]
  const uint32_t redbar = sbase + Cfg::OFF_REDBAR;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = static_cast<int>(blockIdx.x) % p.splits;   // the cluster rank
  const int n0 = (static_cast<int>(blockIdx.x) / p.splits) * kSkinnyRows;
  const int ks0 = split * p.ks_per_cta;
  const int ks1 = min(ks0 + p.ks_per_cta, p.num_ks);
  const int nst = ks1 - ks0;   // >= 1: the host plans no empty split
  // The outputs of the N-block, token-major: E = (valid tokens) x 64.  Rank r
  // owns [cut(r), cut(r + 1)).
  const int S = p.splits;
  const int E = min(p.M, Cfg::A_ROWS) * kSkinnyRows;
  auto cut = [&](int r) { return E * r / S; };
  const int own0 = cut(split);
  const int own1 = cut(split + 1);

  for (int i = threadIdx.x; i < Cfg::A_ROWS * kSkinnyRows; i += Cfg::THREADS) part[i] = 0;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, Cfg::COMPUTE_WARPS);
    }
    mbar_init(redbar, 1);
    fence_mbarrier_init();
    // the bytes the other CTAs will add into this CTA's slice
    if (S > 1) mbar_arrive_expect_tx(redbar, static_cast<uint32_t>((S - 1) * (own1 - own0) * 4));
  }
  if (warp == Cfg::COMPUTE_WARPS && lane == 0) {
    // Start the DRAM reads of the ring's first fill while the previous
    // kernel of the stream drains: into L2 only, which is safe before the
    // dependency wait (see tma_prefetch_l2_2d).
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmA);
    for (int i = 0; i < nst && i < Cfg::STAGES; ++i)
#pragma unroll
      for (int b = 0; b < Cfg::W_BOXES; ++b)
        tma_prefetch_l2_2d(&tmW, (ks0 + i) * kSkinnyK + b * Cfg::BOX_K, n0);
  }
  __syncthreads();
  if (S > 1) cluster_sync_all();   // every CTA's part and mbarriers are set up before any red.async
  pdl_wait();   // weights and codes may come from the previous kernel of the stream

  if (warp == Cfg::COMPUTE_WARPS) {
    // ---- producer: one thread streams the stages through the ring
    if (lane == 0) {
      int issued = 0;
#pragma unroll 1
      for (int i = 0; i < nst; ++i) {
        const int s = i % Cfg::STAGES;
        if (i >= Cfg::STAGES &&
            !mbar_wait(empty0 + 8u * s, static_cast<uint32_t>((i / Cfg::STAGES - 1) & 1), abort_flag))
          break;
        const uint32_t st = sbase + static_cast<uint32_t>(s * Cfg::STAGE_BYTES);
        const uint32_t bar = full0 + 8u * s;
        mbar_arrive_expect_tx(bar, Cfg::STAGE_BYTES);
        const int k0 = (ks0 + i) * kSkinnyK;
#pragma unroll
        for (int b = 0; b < Cfg::W_BOXES; ++b)
          tma_load_2d(st + b * Cfg::W_BOX_BYTES, &tmW, bar, k0 + b * Cfg::BOX_K, n0);
#pragma unroll
        for (int b = 0; b < Cfg::A_BOXES; ++b)
          tma_load_2d(st + Cfg::W_BOXES * Cfg::W_BOX_BYTES + b * Cfg::A_BOX_BYTES, &tmA, bar,
                      k0 + b * 128, 0);
        issued = i + 1;
        // keep a second ring's worth of weights on its way into L2 (no
        // shared memory needed), doubling the bytes in flight
        if (i + Cfg::STAGES < nst) {
#pragma unroll
          for (int b = 0; b < Cfg::W_BOXES; ++b)
            tma_prefetch_l2_2d(&tmW, (ks0 + i + Cfg::STAGES) * kSkinnyK + b * Cfg::BOX_K, n0);
        }
      }
      if (*abort_flag) {
        // copies still in flight land before the CTA leaves (bounded)
#pragma unroll 1
        for (int i = issued > Cfg::STAGES ? issued - Cfg::STAGES : 0; i < issued; ++i)
          mbar_wait_bounded(full0 + 8u * (i % Cfg::STAGES),
                            static_cast<uint32_t>((i / Cfg::STAGES) & 1), 100000000ull);
      }
    }
  } else {
    // ---- compute warps
    const int g = lane >> 2;         // weight row (and token) within an 8-group
    const int q = lane & 3;          // quad lane: codes 4q..4q+3 of each 16-block
    const int rw = (warp & 3) * 16;  // the warp's first weight row
    const int h = warp >> 2;         // the warp's K-half of every stage
    float d[MT][kCh][4];
    int acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[t][e] = 0;
#pragma unroll
        for (int c = 0; c < kCh; ++c) d[t][c][e] = 0.0f;
      }
    if (warp == Cfg::COMPUTE_WARPS - 1 && p.out_mode == kOutBf16) {
      // the epilogue's constants, fetched while the first stage streams in
      for (int r = lane; r < kSkinnyRows; r += 32) {
        const int n = min(n0 + r, p.N - 1);
        scl_w[r] = p.s_w[n];
        scl_b[r] = p.bias ? __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16) : 0.0f;
      }
      if (lane < Cfg::A_ROWS) scl_a[lane] = p.s_a[min(lane, p.M - 1)];
    }
    bool ok = true;
#pragma unroll 1
    for (int i = 0; i < nst; ++i) {
      const int s = i % Cfg::STAGES;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8u * s,
                                             static_cast<uint32_t>((i / Cfg::STAGES) & 1), abort_flag));
      if (!ok) break;
      const uint32_t st = sbase + static_cast<uint32_t>(s * Cfg::STAGE_BYTES);
      const uint32_t abox = st + Cfg::W_BOXES * Cfg::W_BOX_BYTES + h * Cfg::A_BOX_BYTES;
      // all of this half-stage's operand words first (8 K-blocks of 16), then
      // the conversions and MMAs
      uint32_t wlo[8][2], whi[8][2], x[8][MT];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if constexpr (W16) {
          // fp16 codes: K-block j of half h is in box 2h + j / 4, 16-byte
          // chunk 2 (j % 4) + q / 2, bytes 8 (q % 2) .. + 8
          const uint32_t wbox = st + static_cast<uint32_t>((2 * h + (j >> 2)) * Cfg::W_BOX_BYTES);
          const uint32_t off = ((static_cast<uint32_t>(2 * (j & 3) + (q >> 1)) ^ g) << 4) + 8u * (q & 1);
          const uint2 lo = lds64(wbox + (rw + g) * 128u + off);
          const uint2 hi = lds64(wbox + (rw + g + 8) * 128u + off);
          wlo[j][0] = lo.x;
          wlo[j][1] = lo.y;
          whi[j][0] = hi.x;
          whi[j][1] = hi.y;
        } else {
          // int8 codes: K-block j of half h is 16-byte chunk j of box h
          const uint32_t wbox = st + static_cast<uint32_t>(h * Cfg::W_BOX_BYTES);
          const uint32_t off = ((static_cast<uint32_t>(j) ^ g) << 4) + 4u * q;
          wlo[j][0] = lds32(wbox + (rw + g) * 128u + off);
          whi[j][0] = lds32(wbox + (rw + g + 8) * 128u + off);
        }
#pragma unroll
        for (int t = 0; t < MT; ++t)
          x[j][t] = lds32(abox + (8 * t + g) * 128u + ((static_cast<uint32_t>(j) ^ g) << 4) + 4u * q);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8u * s);   // the words are in registers: free the stage
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t a0, a1, a2, a3;
        if constexpr (W16) {
          a0 = wlo[j][0];
          a2 = wlo[j][1];
          a1 = whi[j][0];
          a3 = whi[j][1];
        } else {
          s8x4_to_f16x4(wlo[j][0], a0, a2);
          s8x4_to_f16x4(whi[j][0], a1, a3);
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          uint32_t b0, b1;
          s8x4_to_f16x4(x[j][t], b0, b1);
          mma_m16n8k16_f16(d[t][j % kCh], a0, a1, a2, a3, b0, b1);
        }
      }
      if (i % kDrainStages == kDrainStages - 1 || i == nst - 1) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v = d[t][0][e];
#pragma unroll
            for (int c = 1; c < kCh; ++c) v = __fadd_rn(v, d[t][c][e]);   // exact (integers < 2^24)
            acc[t][e] += f32_exact_int_to_s32(__float_as_uint(v));
#pragma unroll
            for (int c = 0; c < kCh; ++c) d[t][c][e] = 0.0f;
          }
      }
    }
    // D fragment: e = 0, 1 -> weight row g, tokens 2q, 2q + 1 of group t;
    // e = 2, 3 -> weight row g + 8.  part is token-major: [token][row].
    if (ok) {
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int token = 8 * t + 2 * q + (e & 1);
          const int row = rw + g + (e >= 2 ? 8 : 0);
          if (acc[t][e] != 0) atomicAdd(part + token * kSkinnyRows + row, acc[t][e]);
        }
    }
  }
  pdl_trigger();
  __syncthreads();
  if (S > 1) {
    // Add this CTA's partials of the other owners' slices into theirs
    // (always, so that no owner waits in vain), then wait for the other
    // CTAs' partials of the slice this CTA owns.
    for (int e = static_cast<int>(threadIdx.x); e < E; e += Cfg::THREADS) {
      if (e >= own0 && e < own1) continue;
      int r = 0;   // the owner of value e
      for (int rr = 1; rr < S; ++rr)
        if (cut(rr) <= e) r = rr;
      red_async_add_s32(mapa_shared(smem_u32(part + e), static_cast<uint32_t>(r)), part[e],
                        mapa_shared(redbar, static_cast<uint32_t>(r)));
    }
    mbar_wait_cluster(redbar, 0u, abort_flag);
  }
  const bool write = *abort_flag == 0;
  for (int e = own0 + static_cast<int>(threadIdx.x); e < own1; e += Cfg::THREADS) {
    const int m = e / kSkinnyRows;
    const int r = e % kSkinnyRows;
    const int n = n0 + r;
    if (n >= p.N || !write) continue;
    const int v = part[e];
    if (p.out_mode == kOutBf16) {
      const __nv_bfloat16 y = __float2bfloat16_rn(dequant_one(v, scl_a[m], scl_w[r], scl_b[r]));
      static_cast<uint16_t*>(p.out)[static_cast<int64_t>(m) * p.ldo + n] =
          *reinterpret_cast<const uint16_t*>(&y);
    } else {
      static_cast<int32_t*>(p.out)[static_cast<int64_t>(m) * p.ldo + n] = v;
    }
  }
}

}  // namespace i8
