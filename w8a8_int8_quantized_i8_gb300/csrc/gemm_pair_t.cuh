// gemm_pair_t.cuh -- the fused W8A8 GEMM on a CTA pair with A held in TMEM.
//
// Same arithmetic as gemm.cuh / gemm_pair.cuh (int8 codes through the fp16
// tensor pipe, exact chunked accumulation, fused per-token x per-channel
// dequant + bias; Fused INT8 GEMM Kernel for Ideogram 4.0, arXiv 2606.14598,
// abstract).  Differences from gemm_pair.cuh:
//   * the widened activation codes never touch shared memory: converter warps
//     read the int8 tile, widen it in registers and write it into tensor
//     memory (tcgen05.st); tcgen05.mma.cta_group::2 reads A from TMEM and
//     only W from shared memory.  That removes A's fp16 store and the MMA's
//     read of it from the shared-memory budget per K step;
//   * pair tiles are 256 x 192 so that two fp32 accumulators (2 x 192 TMEM
//     columns) and four A stages (4 x 32 columns) fit in the 512 columns.
// TMEM columns per CTA: D0 [0, 192), D1 [192, 384), A stage s [384 + 32 s, +32).
// A stage layout: lane = row of this CTA's 128 activation rows, column j holds
// codes 2j (low half) and 2j + 1 (high half) of the 64-wide K stage.
#pragma once
#include "gemm_pair.cuh"

namespace i8 {

template <int S8_, int S16_, bool CONV_B_>
struct PairTCfg {
  static constexpr int BM = 128;        // A rows per CTA (TMEM lanes)
  static constexpr int BNH = 96;        // W rows staged per CTA
  static constexpr int PAIR_M = 256;
  static constexpr int PAIR_N = 192;
  static constexpr int S8 = S8_;
  static constexpr int S16 = S16_;
  static constexpr bool CONV_B = CONV_B_;
  static constexpr int BK8 = 128;
  static constexpr int BK16 = 64;
  static constexpr int EPI_WARPS = 8;   // 4 lane quarters x 2 column groups of 96
  static constexpr int EPI_WARP0 = 8;
  static constexpr int THREADS = 512;
  static constexpr int REG_LO = 96;
  static constexpr int REG_HI = 160;
  static_assert(2 * 128 * REG_LO + 2 * 128 * REG_HI <= THREADS * (65536 / THREADS),
                "register split exceeds the launch allocation");
  static constexpr int A8_BYTES = BM * BK8;                      // 16 KB
  static constexpr int B8_BYTES = CONV_B ? BNH * BK8 : 0;        // 12 KB
  static constexpr int STAGE8 = A8_BYTES + B8_BYTES;
  static constexpr int B16_BYTES = BNH * BK16 * 2;               // 12 KB
  static constexpr int OFF_S8 = 0;
  static constexpr int OFF_S16 = OFF_S8 + S8 * STAGE8;
  static constexpr int OFF_EPI = OFF_S16 + S16 * B16_BYTES;
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * 4096;
  static constexpr int NUM_BARS = 2 * S8 + 4 * S16 + 7;          // same set as PairBars
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TMEM_COLS = 512;
  static constexpr int TMEM_A0 = 2 * PAIR_N;                     // 384
  static constexpr uint32_t TX8 = STAGE8;
  static constexpr uint32_t TX16 = CONV_B ? 0 : B16_BYTES;
  // W conversion items (16-byte int8 chunks) per fp16 stage: 96 rows x 4.
  // Warps 2-3 take four each, warps 4-7 (which also widen A) one each.
  static constexpr int B_ITEMS = CONV_B ? BNH * 4 : 0;
  static_assert(S8 * STAGE8 % 1024 == 0 && B16_BYTES % 1024 == 0, "stage alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(TMEM_A0 + 32 * S16 <= TMEM_COLS, "tensor memory");
};

// D (+)= A[tmem] * B[smem]^T across the CTA pair (A rows from each CTA's TMEM
// at the same address, B rows from each CTA's shared memory).
__device__ __forceinline__ void mma_f16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Store one warp's 32 rows x COLS columns in 32-column groups through a
// 4 KB staging buffer and bulk tensor stores: bf16 rows of 64 bytes with the
// 64-byte swizzle (chunk c of row r at c ^ ((r >> 1) & 3)), int32 rows of
// 128 bytes with the 128-byte swizzle.  tmY boxes are 32 x 32.
template <int COLS>
__device__ __forceinline__ void store_warp_tile_g32(const GemmParams& p, const CUtensorMap* tmY,
                                                    uint32_t stage, int lane, int m_base, int n0,
                                                    const int (&acc)[COLS], int z) {
  const int m = m_base + lane;
  if (p.out_mode == kOutBf16) {
    const uint32_t row = stage + static_cast<uint32_t>(lane) * 64u;
    const uint32_t x = static_cast<uint32_t>((lane >> 1) & 3);
    const float sa = m < p.M ? p.s_a[m] : 0.0f;
    const unsigned long long sa2 = f2(sa, sa);
#pragma unroll
    for (int g = 0; g < COLS / 32; ++g) {
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      const int nb = n0 + g * 32;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
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
          const int j = g * 32 + 8 * c + 2 * i;
          unsigned long long t = f2(__int2float_rn(acc[j]), __int2float_rn(acc[j + 1]));
          t = f2_mul(t, sa2);
          t = f2_mul(t, f2(sw[2 * i], sw[2 * i + 1]));
          t = f2_add(t, f2(__uint_as_float(bw[i] << 16), __uint_as_float(bw[i] & 0xFFFF0000u)));
          float lo, hi;
          f2_split(t, lo, hi);
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
  } else {
    const uint32_t row = stage + static_cast<uint32_t>(lane) * 128u;
    const uint32_t x = static_cast<uint32_t>(lane & 7);
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
        tma_store_3d(tmY, stage, n0 + g * 32, m_base, z);
        bulk_commit_group();
      }
    }
  }
}

template <class Cfg>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg::THREADS, 1)
    gemm_w8a8_pair_t_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  const PairBars bars{sbase + Cfg::OFF_BAR, Cfg::S8, Cfg::S16};
  auto stage8 = [&](int s) { return sbase + Cfg::OFF_S8 + static_cast<uint32_t>(s * Cfg::STAGE8); };
  auto stage16 = [&](int s) { return sbase + Cfg::OFF_S16 + static_cast<uint32_t>(s * Cfg::B16_BYTES); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::S8; ++s) {
      mbar_init(bars.full8(s), 1);
      mbar_init(bars.empty8(s), 6);                 // converter warps 2..7
    }
    for (int s = 0; s < Cfg::S16; ++s) {
      mbar_init(bars.full16(s), 6);
      mbar_init(bars.tma16(s), 1);
      mbar_init(bars.empty16(s), 1);
      mbar_init(bars.pfull16(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.accfull(b), 1);
      mbar_init(bars.accempty(b), Cfg::EPI_WARPS);
      mbar_init(bars.paccempty(b), 1);
    }
    mbar_init(bars.done(), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
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
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp >= Cfg::EPI_WARP0) {
    regs_inc<Cfg::REG_HI>();
    // ------------------------------------------------------------ epilogue
    const int ew = warp - Cfg::EPI_WARP0;
    const int quarter = warp & 3;
    const int cg = ew >> 2;                 // 96-column group
    Ring racc;
    bool ok = true;
    for (int tile = pair; ok && tile < p.num_tiles; tile += npairs) {
      const PairTile tc = decode_pair_tile(p, tile);
      const int nst = 2 * (tc.kb1 - tc.kb0);
      int acc[96];
#pragma unroll
      for (int i = 0; i < 96; ++i) acc[i] = 0;
      for (int st0 = 0; st0 < nst; st0 += p.chunk_stages) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.accfull(racc.s), racc.ph, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(racc.s * Cfg::PAIR_N + cg * 96);
#pragma unroll
        for (int q3 = 0; q3 < 3; ++q3) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + q3 * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[q3 * 32 + i] += f32_exact_int_to_s32(r[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.accempty(racc.s));
        racc.advance(2);
      }
      if (!ok) break;
      const uint32_t stg = sbase + Cfg::OFF_EPI + static_cast<uint32_t>(ew) * 4096u;
      store_warp_tile_g32<96>(p, &tmY, stg, lane,
                              tc.mp * Cfg::PAIR_M + static_cast<int>(rank) * Cfg::BM + quarter * 32,
                              tc.nb * Cfg::PAIR_N + cg * 96, acc, tc.ks);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else if (warp == 0) {
    regs_dec<Cfg::REG_LO>();
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Ring r8, r16;
      bool ok = true;
      for (int tile = pair; ok && tile < p.num_tiles; tile += npairs) {
        const PairTile tc = decode_pair_tile(p, tile);
        const int m0 = tc.mp * Cfg::PAIR_M + static_cast<int>(rank) * Cfg::BM;
        const int n0 = tc.nb * Cfg::PAIR_N + static_cast<int>(rank) * Cfg::BNH;
        for (int kb = tc.kb0; ok && kb < tc.kb1; ++kb) {
          if (!(ok = mbar_wait(bars.empty8(r8.s), r8.ph ^ 1u, abort_flag))) break;
          mbar_arrive_expect_tx(bars.full8(r8.s), Cfg::TX8);
          tma_load_2d(stage8(r8.s), &tmA, bars.full8(r8.s), kb * Cfg::BK8, m0);
          if constexpr (Cfg::CONV_B)
            tma_load_2d(stage8(r8.s) + Cfg::A8_BYTES, &tmB, bars.full8(r8.s), kb * Cfg::BK8, n0);
          r8.advance(Cfg::S8);
          if constexpr (!Cfg::CONV_B) {
            for (int h = 0; h < 2; ++h) {
              if (!(ok = mbar_wait(bars.empty16(r16.s), r16.ph ^ 1u, abort_flag))) break;
              mbar_arrive_expect_tx(bars.tma16(r16.s), Cfg::TX16);
              tma_load_2d(stage16(r16.s), &tmB, bars.tma16(r16.s), kb * Cfg::BK8 + h * Cfg::BK16, n0);
              r16.advance(Cfg::S16);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    regs_dec<Cfg::REG_LO>();
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(Cfg::PAIR_M, Cfg::PAIR_N);
      Ring r16, racc;
      bool ok = true;
      for (int tile = pair; ok && tile < p.num_tiles; tile += npairs) {
        const PairTile tc = decode_pair_tile(p, tile);
        const int nst = 2 * (tc.kb1 - tc.kb0);
        for (int st0 = 0; ok && st0 < nst; st0 += p.chunk_stages) {
          const int st1 = min(nst, st0 + p.chunk_stages);
          if (!(ok = mbar_wait(bars.accempty(racc.s), racc.ph ^ 1u, abort_flag))) break;
          if (!(ok = mbar_wait(bars.paccempty(racc.s), racc.ph ^ 1u, abort_flag))) break;
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(racc.s * Cfg::PAIR_N);
          for (int st = st0; st < st1; ++st) {
            if (!(ok = mbar_wait(bars.full16(r16.s), r16.ph, abort_flag))) break;
            if (!(ok = mbar_wait(bars.pfull16(r16.s), r16.ph, abort_flag))) break;
            tc_fence_after();
            const uint32_t a = tmem_base + static_cast<uint32_t>(Cfg::TMEM_A0 + 32 * r16.s);
            const uint64_t bd = smem_desc_sw128(stage16(r16.s));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              mma_f16_ts_pair(d, a + 8u * j, bd + 2u * j, idesc, (st > st0 || j > 0) ? 1u : 0u);
            }
            mma_commit_pair(bars.empty16(r16.s), 0x3);
            r16.advance(Cfg::S16);
          }
          if (!ok) break;
          mma_commit_pair(bars.accfull(racc.s), 0x3);
          racc.advance(2);
        }
      }
      mma_commit_pair(bars.done(), 0x1);
      mbar_wait_bounded(bars.done(), 0u, 100000000ull);
    } else if (lane == 0) {
      // ---------------------------------------------------------- relay (CTA 1)
      const uint32_t pfull0 = mapa_shared(bars.pfull16(0), 0);
      const uint32_t pacc0 = mapa_shared(bars.paccempty(0), 0);
      Ring r16, racc;
      int chunk = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < p.num_tiles; tile += npairs) {
        const PairTile tc = decode_pair_tile(p, tile);
        const int nst = 2 * (tc.kb1 - tc.kb0);
        for (int st0 = 0; ok && st0 < nst; st0 += p.chunk_stages, ++chunk) {
          const int st1 = min(nst, st0 + p.chunk_stages);
          if (chunk >= 2) {
            if (!(ok = mbar_wait(bars.accempty(racc.s), racc.ph ^ 1u, abort_flag))) break;
            mbar_arrive_remote_cta(pacc0 + 8u * racc.s);
          }
          racc.advance(2);
          for (int st = st0; st < st1; ++st) {
            if (!(ok = mbar_wait(bars.full16(r16.s), r16.ph, abort_flag))) break;
            mbar_arrive_remote_cta(pfull0 + 8u * r16.s);
            r16.advance(Cfg::S16);
          }
        }
      }
    }
  } else {
    regs_dec<Cfg::REG_LO>();
    // ------------------------------------------------------------ converters (warps 2..7)
    const bool a_warp = warp >= 4;
    const int arow = 32 * (warp & 3) + lane;            // A row == TMEM lane
    const uint32_t a_lane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    // W items: warps 2-3 -> 4 each (items ct + 64 j), warps 4-7 -> one (256 + ct')
    constexpr int BIPT = 4;
    ConvItem bitems[BIPT];
    int nb_items = 0;
    if constexpr (Cfg::CONV_B) {
      const int ct = threadIdx.x - 64;                  // 0..191
#pragma unroll
      for (int j = 0; j < BIPT; ++j) {
        int i = -1;
        if (!a_warp) i = ct + 64 * j;                   // 0..255
        else if (j == 0) i = 256 + (ct - 64);           // 256..383
        if (i >= 0 && i < Cfg::B_ITEMS) {
          const int cl = i / Cfg::BNH;
          const int r = i % Cfg::BNH;
          const int x = r & 7;
          bitems[j].src = static_cast<uint32_t>(Cfg::A8_BYTES + r * 128 + ((cl ^ x) << 4));
          bitems[j].dst = static_cast<uint32_t>(r * 128 + (((2 * cl) ^ x) << 4));
          nb_items = j + 1;
        }
      }
    }
    Ring r8, r16;
    bool ok = true;
    for (int tile = pair; ok && tile < p.num_tiles; tile += npairs) {
      const PairTile tc = decode_pair_tile(p, tile);
      for (int kb = tc.kb0; kb < tc.kb1; ++kb) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.full8(r8.s), r8.ph, abort_flag));
        if (!ok) break;
        const uint32_t s8 = stage8(r8.s);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          // int8 inputs of this K-half: W items and (A warps) 4 chunks of the row
          uint4 bv[BIPT];
#pragma unroll
          for (int j = 0; j < BIPT; ++j)
            if (j < nb_items) bv[j] = lds128(s8 + (bitems[j].src ^ (static_cast<uint32_t>(h) << 6)));
          uint4 av[4];
          if (a_warp) {
            const uint32_t arow_addr = s8 + static_cast<uint32_t>(arow) * 128u;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              av[c] = lds128(arow_addr + ((((h << 2) | c) ^ (arow & 7)) << 4));
          }
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.empty16(r16.s), r16.ph ^ 1u, abort_flag));
          if (!ok) break;
          if constexpr (Cfg::CONV_B) {
            const uint32_t s16 = stage16(r16.s);
#pragma unroll
            for (int j = 0; j < BIPT; ++j) {
              if (j < nb_items) {
                uint4 o0, o1;
                s8x4_to_f16x4(bv[j].x, o0.x, o0.y);
                s8x4_to_f16x4(bv[j].y, o0.z, o0.w);
                s8x4_to_f16x4(bv[j].z, o1.x, o1.y);
                s8x4_to_f16x4(bv[j].w, o1.z, o1.w);
                sts128(s16 + bitems[j].dst, o0);
                sts128(s16 + (bitems[j].dst ^ 16u), o1);
              }
            }
            fence_proxy_async_smem();
          }
          if (a_warp) {
            uint32_t t[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              s8x4_to_f16x4(av[c].x, t[8 * c + 0], t[8 * c + 1]);
              s8x4_to_f16x4(av[c].y, t[8 * c + 2], t[8 * c + 3]);
              s8x4_to_f16x4(av[c].z, t[8 * c + 4], t[8 * c + 5]);
              s8x4_to_f16x4(av[c].w, t[8 * c + 6], t[8 * c + 7]);
            }
            tmem_st_32x32b_x32(tmem_base + a_lane + static_cast<uint32_t>(Cfg::TMEM_A0 + 32 * r16.s), t);
            tmem_wait_st();
          }
          if constexpr (!Cfg::CONV_B) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.tma16(r16.s), r16.ph, abort_flag));
            if (!ok) break;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.full16(r16.s));
          r16.advance(Cfg::S16);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.empty8(r8.s));
        r8.advance(Cfg::S8);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace i8
