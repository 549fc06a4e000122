// gemm_direct.cuh -- the converter-free CTA-pair GEMM: operands go from HBM
// to shared memory by TMA and straight into tcgen05.mma, nothing is widened
// on chip.  Two modes of one kernel template:
//
// * E4M3 (the FP8 arm).  Fused INT8 GEMM Kernel for Ideogram 4.0 (arXiv
//   2606.14598), abstract: the INT8 kernel is measured against an FP8
//   baseline, and on B200 it loses to the card's native FP8 path.  This is
//   that native path on sm_103a, with the same per-token x per-channel scales
//   and the same fused epilogue:
//     acc[m,n] = sum_k a[m,k] * w[n,k]    (E4M3 x E4M3 -> fp32, kind::f8f6f4)
//     y[m,n]   = bf16(acc * s_a[m] * s_w[n] + bias[n])
//   The tensor core's fp32 additions round (in an order the hardware does not
//   specify), so this mode agrees with the exact oracle within an error bound.
//
// * F16 codes (the exact W8A8 path without on-chip widening).  The same
//   int8 x int8 -> int32 product as gemm.cuh / gemm_pair.cuh, with both
//   operands' int8 codes stored as fp16 values of the same integers (the
//   quantizer's fp16-code output, and weights widened once offline).
//   kind::f16 products are exact, and the fp32 accumulator is restarted every
//   `chunk` K so that no partial sum reaches 2^24; the epilogue warps drain
//   each chunk into int32 registers.  Bit-exact, like the int8-code kernels.
//
// Structure: the two CTAs of a cluster compute one 256 x 256 output tile.
//   * CTA r loads A rows [m0 + 128 r, +128) and B rows [n0 + 128 r, +128) of
//     each 128-byte-deep K block (128 E4M3 or 64 fp16 codes) into its own
//     shared memory (128-byte swizzle); both CTAs' loads complete on CTA 0's
//     full barrier (cta_group::2 TMA), which CTA 0's producer armed with the
//     stage's total byte count.
//   * One thread of CTA 0 issues four M=256 N=256 MMAs per block (K = 32 E4M3
//     or 16 fp16 codes each, 32 bytes along the swizzled row); each CTA's 128
//     rows x 256 fp32 columns land in its own tensor memory, in one of two
//     buffers, so the epilogue overlaps the next MMAs.  Its commits free the
//     stage in both CTAs (multicast).
//   * Eight epilogue warps per CTA (lane quarter = warp % 4, column half =
//     (warp - 4) / 4) read the accumulator, hand the buffer back (CTA 1's
//     warps arrive on CTA 0's barrier), and write the tile through swizzled
//     shared-memory staging with bulk tensor stores: dequant + bias -> bf16,
//     or the raw accumulator (fp32 / int32) for the checking paths.
// Warps: 0 producer, 1 TMEM allocation + MMA issuer, 2-3 idle, 4-11 epilogue;
// setmaxnreg moves registers from warpgroup 0 to the epilogue warpgroups.
// With few tiles (small M or N) the K range is split: each (tile, split) item
// writes a partial into a workspace plane, and a fix-up kernel adds the
// planes in split order (fp32 for E4M3, exact int32 for F16 codes) and
// applies the epilogue.
// Every wait is bounded (ptx.cuh); a timeout aborts the CTA cleanly.
#pragma once
#include "gemm.cuh"

namespace i8 {

enum DirectKind : int { kDirectE4M3 = 0, kDirectF16 = 1 };

template <int KIND>
struct DirectCfg {
  static constexpr int BM = 128;        // A rows loaded per CTA
  static constexpr int BN = 128;        // B rows loaded per CTA
  static constexpr int PAIR_M = 256;
  static constexpr int PAIR_N = 256;
  static constexpr int BK = KIND == kDirectF16 ? 64 : 128;   // K per stage: one 128-byte row
  static constexpr int STAGES = 6;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_WARP0 = 4;
  static constexpr int THREADS = 384;
  // registers per thread after setmaxnreg: warpgroup 0 (producer, MMA
  // issuer, two idle warps) hands registers to the two epilogue warpgroups
  static constexpr int REG_LO = 136;
  static constexpr int REG_HI = 176;
  static_assert(128 * REG_LO + 256 * REG_HI <= THREADS * ((65536 / THREADS) & ~7),
                "register split exceeds the launch allocation");
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_EPI = STAGES * STAGE_BYTES;          // 4 KB staging per epilogue warp
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * 4096;
  // full[S] empty[S] accfull[2] accempty[2] done sclfull sclfree
  static constexpr int NUM_BARS = 2 * STAGES + 7;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  // the current tile's per-channel scales (fp32) and bias (bf16), staged by
  // the epilogue warps: PAIR_N columns
  static constexpr int OFF_SCL = (OFF_MISC + 16 + 15) / 16 * 16;
  static constexpr int OFF_SCL_BIAS = OFF_SCL + PAIR_N * 4;
  static constexpr int SMEM_BYTES = OFF_SCL_BIAS + PAIR_N * 2 + 1024;
  static constexpr int TMEM_COLS = 2 * PAIR_N;
  static constexpr uint32_t TX = 2 * STAGE_BYTES;               // both CTAs' loads of a stage
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
};

// Work item `item` of the schedule: K split ks of tile (mp, nb); the tile's
// tiles run in tile_coords order (M or N blocks fastest, by the host's choice).
struct DirectItem {
  int mp, nb, ks, kb0, kb1;
};
__device__ __forceinline__ DirectItem direct_item(const GemmParams& p, int item) {
  DirectItem t;
  t.ks = item % p.splits;
  const int tile = item / p.splits;
  tile_coords(p, tile, t.mp, t.nb);
  t.kb0 = t.ks * p.kb_per_split;
  t.kb1 = min(t.kb0 + p.kb_per_split, p.total_kb);
  return t;
}

template <int STAGES>
struct DirectBars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8u * s; }
  __device__ uint32_t empty(int s) const { return base + 8u * (STAGES + s); }
  __device__ uint32_t accfull(int b) const { return base + 8u * (2 * STAGES + b); }
  __device__ uint32_t accempty(int b) const { return base + 8u * (2 * STAGES + 2 + b); }
  __device__ uint32_t done() const { return base + 8u * (2 * STAGES + 4); }
  __device__ uint32_t sclfull() const { return base + 8u * (2 * STAGES + 5); }
  __device__ uint32_t sclfree() const { return base + 8u * (2 * STAGES + 6); }
};

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DirectCfg<KIND>::THREADS, 1)
    gemm_direct_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
  using Cfg = DirectCfg<KIND>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  const DirectBars<Cfg::STAGES> bars{sbase + Cfg::OFF_BAR};
  auto stage = [&](int s) { return sbase + Cfg::OFF_STAGE + static_cast<uint32_t>(s * Cfg::STAGE_BYTES); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(bars.full(s), 1);        // CTA 0: its producer's arrive + both CTAs' bytes
      mbar_init(bars.empty(s), 1);       // the MMA thread's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.accfull(b), 1);
      mbar_init(bars.accempty(b), 2 * Cfg::EPI_WARPS);  // CTA 0: both CTAs' epilogue warps
    }
    mbar_init(bars.done(), 1);
    mbar_init(bars.sclfull(), Cfg::EPI_WARPS);
    mbar_init(bars.sclfree(), Cfg::EPI_WARPS);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp >= 2 && lane == 0) {
    // The first read of a launch parameter misses the constant cache (about
    // 1 us on GB300) and would sit on every role's path to its first tile;
    // touch the fields the roles decode first while warps 0 and 1 set up the
    // barriers and the tensor memory.
    const int t = p.num_tiles ^ p.splits ^ p.total_kb ^ p.kb_per_split ^ p.num_m_blk ^
                  p.num_n_blk ^ p.n_fastest ^ p.chunk_stages ^ p.out_mode ^ p.M ^ p.N ^
                  static_cast<int>(reinterpret_cast<uintptr_t>(p.s_a)) ^
                  static_cast<int>(reinterpret_cast<uintptr_t>(p.s_w));
    asm volatile("" ::"r"(t));
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmY);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // operands and outputs may belong to the previous kernel

  if (warp == 0) {
    regs_dec<Cfg::REG_LO>();
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(bars.full(0), 0);
      Ring r;
      bool ok = true;
      const int items = p.num_tiles * p.splits;
      for (int item = pair; ok && item < items; item += npairs) {
        const DirectItem t = direct_item(p, item);
        const int m0 = t.mp * Cfg::PAIR_M + static_cast<int>(rank) * Cfg::BM;
        const int n0 = t.nb * Cfg::PAIR_N + static_cast<int>(rank) * Cfg::BN;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!(ok = mbar_wait(bars.empty(r.s), r.ph ^ 1u, abort_flag))) break;
          if (rank == 0) mbar_arrive_expect_tx(bars.full(r.s), Cfg::TX);
          const uint32_t fb = full0 + 8u * static_cast<uint32_t>(r.s);
          tma_load_2d_pair(stage(r.s), &tmA, fb, kb * Cfg::BK, m0);
          tma_load_2d_pair(stage(r.s) + Cfg::A_BYTES, &tmB, fb, kb * Cfg::BK, n0);
          r.advance(Cfg::STAGES);
        }
      }
    }
  } else if (warp == 1) {
    regs_dec<Cfg::REG_LO>();
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = KIND == kDirectF16 ? idesc_f16_f32(Cfg::PAIR_M, Cfg::PAIR_N)
                                                    : idesc_e4m3_f32(Cfg::PAIR_M, Cfg::PAIR_N);
      Ring r, racc;
      bool ok = true;
      const int items = p.num_tiles * p.splits;
      for (int item = pair; ok && item < items; item += npairs) {
        const DirectItem t = direct_item(p, item);
        // F16 codes: the fp32 accumulator restarts every chunk_stages blocks
        // (exactness); E4M3: one accumulation over the item's K range
        const int chunk = KIND == kDirectF16 ? p.chunk_stages : t.kb1 - t.kb0;
        for (int kc = t.kb0; ok && kc < t.kb1; kc += chunk) {
          const int kc1 = min(t.kb1, kc + chunk);
          if (!(ok = mbar_wait_cluster(bars.accempty(racc.s), racc.ph ^ 1u, abort_flag))) break;
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(racc.s * Cfg::PAIR_N);
          for (int kb = kc; kb < kc1; ++kb) {
            if (!(ok = mbar_wait_cluster(bars.full(r.s), r.ph, abort_flag))) break;
            tc_fence_after();
            const uint64_t ad = smem_desc_sw128(stage(r.s));
            const uint64_t bd = smem_desc_sw128(stage(r.s) + Cfg::A_BYTES);
#pragma unroll
            for (int j = 0; j < 4; ++j) {   // 32 bytes of K per MMA along the swizzled row
              const uint32_t accum = (kb > kc || j > 0) ? 1u : 0u;
              if constexpr (KIND == kDirectF16) mma_f16_ss_pair(d, ad + 2u * j, bd + 2u * j, idesc, accum);
              else mma_f8_ss_pair(d, ad + 2u * j, bd + 2u * j, idesc, accum);
            }
            mma_commit_pair(bars.empty(r.s), 0x3);
            r.advance(Cfg::STAGES);
          }
          if (!ok) break;
          mma_commit_pair(bars.accfull(racc.s), 0x3);
          racc.advance(2);
        }
      }
      mma_commit_pair(bars.done(), 0x1);
      mbar_wait_bounded(bars.done(), 0u, 100000000ull);
    }
  } else if (warp >= Cfg::EPI_WARP0) {
    regs_inc<Cfg::REG_HI>();
    // ------------------------------------------------------------ epilogue
    const int ew = warp - Cfg::EPI_WARP0;
    const int quarter = warp & 3;
    const int cg = ew >> 2;
    const uint32_t stage_y = sbase + Cfg::OFF_EPI + static_cast<uint32_t>(ew) * 4096u;
    const uint32_t accempty0 = rank == 0 ? bars.accempty(0) : mapa_shared(bars.accempty(0), 0);
    const bool bf16_out = p.out_mode == kOutBf16;
    const uint32_t scl_w = sbase + Cfg::OFF_SCL;
    const uint32_t scl_b = sbase + Cfg::OFF_SCL_BIAS;
    Ring racc, rscl;
    bool ok = true;
    const int items = p.num_tiles * p.splits;
    for (int item = pair; ok && item < items; item += npairs) {
      const DirectItem t = direct_item(p, item);
      const int chunk = KIND == kDirectF16 ? p.chunk_stages : t.kb1 - t.kb0;
      const int m_base = t.mp * Cfg::PAIR_M + static_cast<int>(rank) * Cfg::BM + quarter * 32;
      float sa = 0.0f;
      if (bf16_out) {
        // Stage this tile's per-channel scales and bias (once the previous
        // tile's readers are done with them) and load this lane's per-token
        // scale while the tile's MMAs run.
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.sclfree(), rscl.ph ^ 1u, abort_flag));
        if (!ok) break;
        stage_channel_scales(p, scl_w, scl_b, t.nb * Cfg::PAIR_N, ew, lane);
        if (m_base + lane < p.M) sa = p.s_a[m_base + lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.sclfull());
      }
      // F16: exact int32 sum of the chunks; E4M3: the fp32 bit patterns
      int acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0;
      for (int kc = t.kb0; kc < t.kb1; kc += chunk) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.accfull(racc.s), racc.ph, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(racc.s * Cfg::PAIR_N + cg * 128);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + q4 * 32, r);
          if constexpr (KIND == kDirectF16) {
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[q4 * 32 + i] += f32_exact_int_to_s32(r[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[q4 * 32 + i] = static_cast<int>(r[i]);
          }
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          const uint32_t bar = accempty0 + 8u * static_cast<uint32_t>(racc.s);
          if (rank == 0) mbar_arrive(bar);
          else mbar_arrive_cluster(bar);
        }
        racc.advance(2);
      }
      if (!ok) break;
      const int n_base = t.nb * Cfg::PAIR_N + cg * 128;
      const int z = p.out_mode == kOutPartial ? t.ks : 0;
      if (bf16_out) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.sclfull(), rscl.ph, abort_flag));
        if (!ok) break;
        // F16 codes: exact int32 sums; E4M3: fp32 accumulator bit patterns
        store_warp_tile_bf16_staged<128, KIND != kDirectF16>(&tmY, stage_y, lane, m_base, n_base,
                                                             acc, sa, scl_w + 4u * (cg * 128),
                                                             scl_b + 2u * (cg * 128));
        // this warp's reads of the staged scales are done
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.sclfree());
        rscl.advance(1);
      } else {
        // int32 (F16 codes) or fp32 (E4M3) accumulators for the checking
        // paths, or a K split's partial in plane ks
        store_warp_tile_s32<128>(&tmY, stage_y, lane, m_base, n_base, acc, z);
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else {
    regs_dec<Cfg::REG_LO>();   // warps 2-3: no role
  }

  __syncwarp();
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's loads, MMAs and remote arrivals are finished
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

// Split-K fix-up of the E4M3 mode (the F16-code mode's int32 partials use
// splitk_reduce_kernel of gemm.cuh): y = epilogue(sum_s partial[s]), the fp32
// partials added in split order (a fixed order, so the result is
// deterministic), then the same fp32 epilogue steps (or the raw sum for the
// checking path).
__global__ void __launch_bounds__(256) splitk_reduce_f32_kernel(const float* __restrict__ ws,
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
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const float* src = ws + static_cast<int64_t>(m) * ldw + n;
    for (int s = 0; s < splits; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(src + s * split_stride);  // ldw % 4 == 0
      acc[0] = __fadd_rn(acc[0], v.x);
      acc[1] = __fadd_rn(acc[1], v.y);
      acc[2] = __fadd_rn(acc[2], v.z);
      acc[3] = __fadd_rn(acc[3], v.w);
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
      float* crow = static_cast<float*>(p.out) + static_cast<int64_t>(m) * p.ldo;
      for (int i = 0; i < cnt; ++i) crow[n + i] = acc[i];
    }
  }
}

}  // namespace i8
