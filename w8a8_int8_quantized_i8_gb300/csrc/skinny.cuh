// skinny.cuh -- the W8A8 GEMM for few tokens (M <= 16), weight streaming.
//
// Same operation as gemm.cuh (Fused INT8 GEMM Kernel for Ideogram 4.0, arXiv
// 2606.14598, abstract: int8 x int8 -> int32, per-token x per-channel dequant
// + bias -> bf16), for the skinny shapes where the weights dominate the bytes
// and the 128-row tensor-core tiles would be almost empty.  KIND selects the
// code formats: int8 weights and tokens; fp16-held weight codes with int8
// tokens; fp16-held codes on both sides (all three exact, int32); or E4M3 on
// both sides (the FP8 arm, fp32 accumulation, m16n8k32 E4M3 MMAs).
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
//   * Eight compute warps: warp w takes the K slice [32 w, 32 w + 32) of
//     every stage for all 64 weight rows, and runs mma.sync m16n8k16 (fp16
//     in, fp32 out) with each 16-row tile of weights as the A operand and
//     the tokens (8, or 16 in two groups) as B.  So every token code is read
//     and widened by one warp only.  Int8 codes for up to 8 tokens skip the
//     widening: the integer m16n8k32 MMA (s8 in, s32 out) takes the codes
//     as they are, exact, at a rate that still outpaces the weight stream
//     for one token group (not for two).  Both operands take the same
//     permutation of K inside each 16-wide block (lane q of a quad reads the
//     4 consecutive codes 4q..4q+3 as one word), which leaves every dot
//     product unchanged.
//   * One fp32 accumulator per (row tile, token group): the four row tiles
//     give consecutive MMAs independent accumulators.  Every 8 stages they
//     are drained into int32 registers.  An MMA covers 16 K, so |partial| <=
//     16 * 127^2 = 258064, and an accumulator gathers at most 16 of them,
//     below 2^22: exact in fp32.  (E4M3: m16n8k32 E4M3 MMAs, fp32 over the
//     whole range.)
//   * The warps' int32 partials meet in shared memory (integer adds).  With
//     one split the CTA applies the epilogue.  With S, cluster rank r owns a
//     slice of about 1/S of the outputs: every other CTA of the cluster adds
//     its partials of that slice into r's (red.async, counted on r's
//     mbarrier), and r applies the epilogue once they are all in.  No global
//     workspace, no atomics in global memory, nothing to clear between
//     calls, and no CTA waits for another except for the partials it owns.
//     E4M3 keeps its sums deterministic instead: each warp writes its fp32
//     partials to its own slab of the idle stage ring, the CTA adds the
//     eight slabs in a fixed order, and the owner adds the cluster's ranks
//     in a fixed order, reading the other CTAs' shared memory between two
//     cluster barriers.
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
constexpr int kDrainStages = 8;       // stages between drains into int32

// Code formats (weights, tokens).
enum SkinnyKind : int {
  kSkI8 = 0,     // int8, int8
  kSkW16 = 1,    // fp16-held int8 codes, int8
  kSkF16 = 2,    // fp16-held int8 codes, fp16-held int8 codes
  kSkE4M3 = 3    // E4M3, E4M3 (fp32 accumulation)
};

template <int KIND, int MT>
struct SkinnyCfg {
  static constexpr bool W_F16 = KIND == kSkW16 || KIND == kSkF16;
  static constexpr bool A_F16 = KIND == kSkF16;
  static constexpr bool FP8 = KIND == kSkE4M3;
  // int8 codes for up to 8 tokens: the integer m16n8k32 MMA straight from
  // the codes (exact int32, nothing to widen); 16 tokens would make its
  // lower rate the limit, so they take the fp16 MMA on widened codes
  static constexpr bool S8MMA = KIND == kSkI8 && MT == 1;
  static constexpr bool K32 = FP8 || S8MMA;                     // m16n8k32 MMAs on 1-byte codes
  // 32-K operand loads by ldmatrix (conflict-free), except E4M3 with one
  // token group, which measured up to 6 % faster with plain 64-bit loads
  static constexpr bool LDSM = K32 && !(FP8 && MT == 1);
  static constexpr int BOX_K = W_F16 ? 64 : 128;                // weight codes per 128-byte row
  static constexpr int W_BOXES = kSkinnyK / BOX_K;              // 2 (1-byte codes) or 4 (fp16)
  static constexpr int W_BOX_BYTES = kSkinnyRows * 128;         // 8 KB
  static constexpr int A_BOX_K = A_F16 ? 64 : 128;              // token codes per 128-byte row
  static constexpr int A_BOXES = kSkinnyK / A_BOX_K;
  static constexpr int A_ROWS = 8 * MT;                         // token rows per box
  static constexpr int A_BOX_BYTES = A_ROWS * 128;
  static constexpr int STAGE_BYTES = W_BOXES * W_BOX_BYTES + A_BOXES * A_BOX_BYTES;
  static constexpr int STAGES = W_F16 ? 4 : (MT == 1 && !FP8 ? 6 : 5);
  static constexpr int COMPUTE_WARPS = 8;
  static constexpr int THREADS = 32 * (COMPUTE_WARPS + 1);    // + the producer warp
  // partials, token-major: int32 [A_ROWS][64] (E4M3: fp32)
  static constexpr int OFF_PART = STAGES * STAGE_BYTES;
  static constexpr int PART_BYTES = A_ROWS * kSkinnyRows * 4;
  static constexpr int OFF_BAR = OFF_PART + PART_BYTES;         // full[STAGES] empty[STAGES]
  static constexpr int OFF_FLAG = OFF_BAR + 2 * STAGES * 8;
  // the epilogue's constants: channel scales and bias (as fp32) of the 64
  // rows, token scales of the A_ROWS tokens
  static constexpr int OFF_SCL = OFF_FLAG + 16;
  // the mbarrier counting the other CTAs' adds into the owned slice
  static constexpr int OFF_REDBAR = (OFF_SCL + (2 * kSkinnyRows + A_ROWS) * 4 + 7) / 8 * 8;
  static constexpr int SMEM_BYTES = OFF_REDBAR + 8 + 1024;   // + 1 KB alignment room
  // two CTAs per SM: 228 KB per SM, 1 KB of it reserved per CTA
  static_assert(W_F16 || 2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs must fit on an SM");
  static_assert(SMEM_BYTES <= 227 * 1024, "more shared memory than a CTA may hold");
  static_assert(!FP8 || COMPUTE_WARPS * A_ROWS * kSkinnyRows * 4 <= OFF_PART,
                "the E4M3 warps' slabs fit in the stage ring");
  static_assert(STAGE_BYTES % 1024 == 0 && W_BOX_BYTES % 1024 == 0 && A_BOX_BYTES % 1024 == 0,
                "128-byte-swizzled boxes must start on 1 KB boundaries");
  // an accumulator gathers two 16-K MMAs per stage between drains
  static_assert(2 * kDrainStages * 16 * 127 * 127 < (1 << 24),
                "fp32 accumulators must stay exact between drains");
};

__device__ __forceinline__ void mma_m16n8k16_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_m16n8k32_e4m3(float (&d)[4], uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint32_t b0,
                                                  uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_m16n8k32_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 32-bit load from shared memory anywhere in the cluster (a mapa_shared
// address).
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// Four (two) 8 x 16-byte matrices from shared memory: lane l gives the
// address of row l % 8 of matrix l / 8, and receives bytes 4 (l % 4) .. + 4
// of row l / 4 of every matrix.
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void ldsm_x2(uint32_t a, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(a));
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

template <int KIND, int MT>
__global__ void __launch_bounds__(SkinnyCfg<KIND, MT>::THREADS)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                       const SkinnyParams p) {
  using Cfg = SkinnyCfg<KIND, MT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);
  const uint32_t full0 = sbase + Cfg::OFF_BAR;
  const uint32_t empty0 = full0 + 8u * Cfg::STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_FLAG);
  int* part = reinterpret_cast<int*>(smem + Cfg::OFF_PART);
  float* partf = reinterpret_cast<float*>(smem + Cfg::OFF_PART);   // E4M3
  float* slab = reinterpret_cast<float*>(smem);   // E4M3, after the last stage: [warp][token][row]
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

  for (int i = threadIdx.x; i < Cfg::PART_BYTES / 4; i += Cfg::THREADS) part[i] = 0;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, Cfg::COMPUTE_WARPS);
    }
    mbar_init(redbar, 1);
    fence_mbarrier_init();
    // the bytes the other CTAs will add into this CTA's slice
    if (S > 1 && !Cfg::FP8) mbar_arrive_expect_tx(redbar, static_cast<uint32_t>((S - 1) * (own1 - own0) * 4));
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
                      k0 + b * Cfg::A_BOX_K, 0);
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
    // ---- compute warps: warp w takes the K slice [32 w, 32 w + 32) of
    // every stage for all 64 weight rows (four row tiles of 16), so every
    // token code is read and widened by one warp only
    const int g = lane >> 2;         // weight row (and token) within an 8-group
    const int q = lane & 3;          // quad lane: codes 4q..4q+3 of each 16-block
    const int w = warp;
    float d[4][MT][4];               // [row tile][token group][fragment]
    int acc[4][MT][4];
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[rt][t][e] = 0;
          d[rt][t][e] = 0.0f;
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
      const uint32_t abase = st + Cfg::W_BOXES * Cfg::W_BOX_BYTES;
      if constexpr (Cfg::K32) {
        // 1-byte codes, 32-K MMAs (E4M3, or int8 for up to 8 tokens):
        // K-block w of 32 is in box w / 4, 16-byte chunks c0 = 2 (w % 4)
        // (K 0..15 of the block) and c0 + 1 (K 16..31).
        const uint32_t c0 = 2u * static_cast<uint32_t>(w & 3);
        const uint32_t wbox = st + static_cast<uint32_t>((w >> 2) * Cfg::W_BOX_BYTES);
        const uint32_t abox = abase + static_cast<uint32_t>((w >> 2) * Cfg::A_BOX_BYTES);
        uint32_t wa[4][4], xb[MT][2];
        if constexpr (Cfg::LDSM) {
          // One ldmatrix.x4 per 16-row weight tile gives the MMA's A
          // fragment as it stands (rows 0-7 and 8-15 of chunk c0, then of
          // c0 + 1); one ldmatrix.x2 per token group gives B.  Each 8-lane
          // group of addresses covers 8 rows at 8 different swizzled chunks:
          // no bank conflicts.
          const uint32_t li = static_cast<uint32_t>(lane & 7);
          const uint32_t a_off = (li + 8u * static_cast<uint32_t>((lane >> 3) & 1)) * 128u +
                                 (((c0 + static_cast<uint32_t>(lane >> 4)) ^ li) << 4);
          const uint32_t b_off = li * 128u + (((c0 + static_cast<uint32_t>((lane >> 3) & 1)) ^ li) << 4);
#pragma unroll
          for (int rt = 0; rt < 4; ++rt)
            ldsm_x4(wbox + static_cast<uint32_t>(16 * rt) * 128u + a_off, wa[rt][0], wa[rt][1], wa[rt][2],
                    wa[rt][3]);
#pragma unroll
          for (int t = 0; t < MT; ++t)
            ldsm_x2(abox + static_cast<uint32_t>(8 * t) * 128u + b_off, xb[t][0], xb[t][1]);
        } else {
          // Lane q of a quad reads codes 8q..8q+7 of its rows: the first
          // four fill the fragment's K slots 4q..4q+3, the last four slots
          // 16+4q..16+4q+3, for the weights and the tokens alike (the same
          // permutation of K on both sides leaves every dot product
          // unchanged).
          const uint32_t off = ((c0 + static_cast<uint32_t>(q >> 1)) ^ static_cast<uint32_t>(g)) << 4 |
                               (8u * static_cast<uint32_t>(q & 1));
#pragma unroll
          for (int rt = 0; rt < 4; ++rt) {
            const uint2 lo = lds64(wbox + (16 * rt + g) * 128u + off);
            const uint2 hi = lds64(wbox + (16 * rt + g + 8) * 128u + off);
            wa[rt][0] = lo.x;
            wa[rt][1] = hi.x;
            wa[rt][2] = lo.y;
            wa[rt][3] = hi.y;
          }
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            const uint2 v = lds64(abox + (8 * t + g) * 128u + off);
            xb[t][0] = v.x;
            xb[t][1] = v.y;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8u * s);   // the words are in registers: free the stage
#pragma unroll
        for (int rt = 0; rt < 4; ++rt)
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            if constexpr (Cfg::FP8)
              mma_m16n8k32_e4m3(d[rt][t], wa[rt][0], wa[rt][1], wa[rt][2], wa[rt][3], xb[t][0], xb[t][1]);
            else   // exact: |sum| <= 127^2 * K < 2^31
              mma_m16n8k32_s8(acc[rt][t], wa[rt][0], wa[rt][1], wa[rt][2], wa[rt][3], xb[t][0], xb[t][1]);
          }
      } else {
        // the slice's two 16-blocks kb = 2w, 2w + 1: all operand words
        // first, then the conversions and MMAs
        uint32_t wlo[2][4][2], whi[2][4][2], x[2][MT][2];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          // fp16 codes: 16-block kb is in box kb / 4, 16-byte chunk
          // 2 (kb % 4) + q / 2, bytes 8 (q % 2) .. + 8; 1-byte codes: in box
          // kb / 8, chunk kb % 8, bytes 4q .. + 4
          const int kb = 2 * w + jj;
          const uint32_t off16 = ((static_cast<uint32_t>(2 * (kb & 3) + (q >> 1)) ^ g) << 4) + 8u * (q & 1);
          const uint32_t off8 = ((static_cast<uint32_t>(kb & 7) ^ g) << 4) + 4u * q;
#pragma unroll
          for (int rt = 0; rt < 4; ++rt) {
            if constexpr (Cfg::W_F16) {
              const uint32_t wbox = st + static_cast<uint32_t>((kb >> 2) * Cfg::W_BOX_BYTES);
              const uint2 lo = lds64(wbox + (16 * rt + g) * 128u + off16);
              const uint2 hi = lds64(wbox + (16 * rt + g + 8) * 128u + off16);
              wlo[jj][rt][0] = lo.x;
              wlo[jj][rt][1] = lo.y;
              whi[jj][rt][0] = hi.x;
              whi[jj][rt][1] = hi.y;
            } else {
              const uint32_t wbox = st + static_cast<uint32_t>((kb >> 3) * Cfg::W_BOX_BYTES);
              wlo[jj][rt][0] = lds32(wbox + (16 * rt + g) * 128u + off8);
              whi[jj][rt][0] = lds32(wbox + (16 * rt + g + 8) * 128u + off8);
            }
          }
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            if constexpr (Cfg::A_F16) {
              const uint32_t abox = abase + static_cast<uint32_t>((kb >> 2) * Cfg::A_BOX_BYTES);
              const uint2 v = lds64(abox + (8 * t + g) * 128u + off16);
              x[jj][t][0] = v.x;
              x[jj][t][1] = v.y;
            } else {
              const uint32_t abox = abase + static_cast<uint32_t>((kb >> 3) * Cfg::A_BOX_BYTES);
              x[jj][t][0] = lds32(abox + (8 * t + g) * 128u + off8);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8u * s);   // the words are in registers: free the stage
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          uint32_t b[MT][2];
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            if constexpr (Cfg::A_F16) {
              b[t][0] = x[jj][t][0];
              b[t][1] = x[jj][t][1];
            } else {
              s8x4_to_f16x4(x[jj][t][0], b[t][0], b[t][1]);
            }
          }
#pragma unroll
          for (int rt = 0; rt < 4; ++rt) {
            uint32_t a0, a1, a2, a3;
            if constexpr (Cfg::W_F16) {
              a0 = wlo[jj][rt][0];
              a2 = wlo[jj][rt][1];
              a1 = whi[jj][rt][0];
              a3 = whi[jj][rt][1];
            } else {
              s8x4_to_f16x4(wlo[jj][rt][0], a0, a2);
              s8x4_to_f16x4(whi[jj][rt][0], a1, a3);
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) mma_m16n8k16_f16(d[rt][t], a0, a1, a2, a3, b[t][0], b[t][1]);
          }
        }
        if (i % kDrainStages == kDrainStages - 1 || i == nst - 1) {
#pragma unroll
          for (int rt = 0; rt < 4; ++rt)
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                acc[rt][t][e] += f32_exact_int_to_s32(__float_as_uint(d[rt][t][e]));
                d[rt][t][e] = 0.0f;
              }
        }
      }
    }
    // E4M3 reuses the ring for its slabs once every compute warp has read
    // its last stage (the producer issues nothing after the last stage)
    if constexpr (Cfg::FP8) named_bar_sync(1, 32 * Cfg::COMPUTE_WARPS);
    // D fragment: e = 0, 1 -> weight row 16 rt + g, tokens 2q, 2q + 1 of
    // group t; e = 2, 3 -> weight row 16 rt + g + 8.  Token-major: [token][row].
    if (ok) {
#pragma unroll
      for (int rt = 0; rt < 4; ++rt)
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int token = 8 * t + 2 * q + (e & 1);
            const int row = 16 * rt + g + (e >= 2 ? 8 : 0);
            if constexpr (Cfg::FP8) {
              // into this warp's own slab of the (now idle) stage ring
              slab[(w * Cfg::A_ROWS + token) * kSkinnyRows + row] = d[rt][t][e];
            } else {
              if (acc[rt][t][e] != 0) atomicAdd(part + token * kSkinnyRows + row, acc[rt][t][e]);
            }
          }
    }
  }
  pdl_trigger();
  __syncthreads();
  if constexpr (Cfg::FP8) {
    // E4M3: this CTA's partials, the eight warps' slabs added in a fixed
    // order; then this CTA's share of the outputs, summed over the
    // cluster's ranks in a fixed order (distributed shared memory, between
    // two cluster barriers).  With one split a thread reads back only the
    // values it wrote.
    for (int e = static_cast<int>(threadIdx.x); e < E; e += Cfg::THREADS) {
      float v = slab[e];
#pragma unroll
      for (int ww = 1; ww < Cfg::COMPUTE_WARPS; ++ww) v = __fadd_rn(v, slab[ww * Cfg::A_ROWS * kSkinnyRows + e]);
      partf[e] = v;
    }
    if (S > 1) cluster_sync_all();   // every CTA's partials are complete and visible
    const bool write = *abort_flag == 0;
    for (int e = own0 + static_cast<int>(threadIdx.x); e < own1; e += Cfg::THREADS) {
      const int m = e / kSkinnyRows;
      const int r = e % kSkinnyRows;
      const int n = n0 + r;
      if (n >= p.N) continue;
      float v;
      if (S > 1) {
        v = 0.0f;
#pragma unroll 1
        for (int rk = 0; rk < S; ++rk)
          v = __fadd_rn(v, ld_shared_cluster_f32(mapa_shared(smem_u32(partf + e), static_cast<uint32_t>(rk))));
      } else {
        v = partf[e];
      }
      if (!write) continue;
      if (p.out_mode == kOutBf16) {
        const __nv_bfloat16 y = __float2bfloat16_rn(dequant_one(v, scl_a[m], scl_w[r], scl_b[r]));
        static_cast<uint16_t*>(p.out)[static_cast<int64_t>(m) * p.ldo + n] =
            *reinterpret_cast<const uint16_t*>(&y);
      } else {
        static_cast<float*>(p.out)[static_cast<int64_t>(m) * p.ldo + n] = v;
      }
    }
    if (S > 1) cluster_sync_all();   // no CTA leaves while another still reads its partials
    return;
  }
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
