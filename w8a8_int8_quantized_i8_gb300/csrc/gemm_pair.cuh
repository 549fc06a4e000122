// gemm_pair.cuh -- the fused W8A8 GEMM on a CTA pair (cta_group::2).
//
// Same arithmetic as gemm.cuh (int8 codes through the fp16 tensor pipe with
// exact chunked accumulation, fused per-token x per-channel dequant + bias).
// Two CTAs of a cluster compute one 256 x 256 output tile together:
//   CTA r (r = 0, 1) stages and widens A rows [m0 + 128 r, +128) and B rows
//   [n0 + 128 r, +128) of every K-block; one thread of CTA 0 issues
//   tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), which reads both
//   CTAs' shared memory and writes each CTA's 128 rows x 256 columns of D
//   into that CTA's tensor memory.  Each SM therefore stages (and widens) half
//   of the B tile it multiplies, which halves the shared-memory traffic per
//   MAC spent on B compared with a 128 x 256 tile on one SM.
// Stages: TMA fills int8 stages of 128 K; converter warps widen each into
// fp16 stages of 64 K, or (WIDE, the default whenever the fp32 chunk is a
// whole number of 128-K stages) one fp16 stage of 128 K made of two 64-K
// swizzled sub-tiles.  Every fp16 stage costs a
// fixed round of hand-offs (converter arrivals, the relay, the MMA thread's
// waits and its commit); at 64 K that round cost as much as the stage's MMAs,
// so the wide stage paid once per 128 K ran 8-14 % faster at DiT shapes.
// Cross-CTA protocol (all waits bounded):
//   * converters arrive on their own CTA's full16[s] and epilogue warps on
//     their own accempty[b] (CTA-scope release: cheap);
//   * in CTA 1 one relay thread forwards each completed phase of those two
//     barriers to CTA 0's pfull16[s] / paccempty[b]: one remote arrive per
//     phase instead of one per warp (a CTA-scope release by default, SYNC
//     below; arrivals straight from CTA 1's warps measured 1-3.5 % slower);
//   * the MMA thread of CTA 0 waits on its own barrier and the forwarded one,
//     and commits to empty16[s] / accfull[b] of both CTAs (multicast).
#pragma once
#include "gemm.cuh"

namespace i8 {

// SYNC selects the memory-model scope of the cross-CTA hand-off:
//   0: relay arrives with release.cluster, the MMA thread waits with acquire.cluster
//   1: relay release.cluster, MMA thread acquire.cta
//   2: relay release.cta (remote arrive), MMA thread acquire.cta
// Measured on GB300 at DiT shapes: 0 and 1 run at ~725 TOPS, 2 at ~920-990
// (the cluster-scope release drains the relay's memory pipeline every stage);
// all three gave bit-exact results on repeated runs.  2 is the default.  The
// data a stage hands over is written to the issuing CTA's own shared memory
// and made visible to the async proxy (fence.proxy.async) before the local
// arrive that the relay observes.
// WIDE_: one fp16 stage holds a whole 128-K int8 block (two 64-K swizzled
// sub-tiles per operand) instead of half of one, so every hand-off (converter
// arrivals, relay, MMA-thread waits and commit) is paid once per 128 K.
template <int S8_, int S16_, bool CONV_A_, bool CONV_B_, int SYNC_ = 2, bool WIDE_ = false>
struct PairCfg {
  static constexpr int SYNC = SYNC_;
  static constexpr bool WIDE = WIDE_;
  static constexpr int K64_PER_STAGE = WIDE ? 2 : 1;   // 64-K sub-tiles per fp16 stage
  static constexpr int BM = 128;        // A rows staged per CTA
  static constexpr int BN = 128;        // B rows staged per CTA
  static constexpr int PAIR_M = 256;
  static constexpr int PAIR_N = 256;
  static constexpr int S8 = S8_;
  static constexpr int S16 = S16_;
  static constexpr bool CONV_A = CONV_A_;
  static constexpr bool CONV_B = CONV_B_;
  static constexpr bool ANY_CONV = CONV_A || CONV_B;
  static constexpr bool ANY_DIRECT = !CONV_A || !CONV_B;
  static constexpr int BK8 = 128;
  static constexpr int BK16 = 64;
  static constexpr int CONV_WARPS = 6;
  static constexpr int CONV_THREADS = CONV_WARPS * 32;
  static constexpr int EPI_WARPS = 8;   // 4 lane quarters x 2 column groups of 128
  static constexpr int EPI_WARP0 = 8;
  static constexpr int NUM_WARPS = 16;
  static constexpr int THREADS = 512;
  static constexpr int REG_LO = 80;
  static constexpr int REG_HI = 176;
  static_assert(2 * 128 * REG_LO + 2 * 128 * REG_HI <= THREADS * (65536 / THREADS),
                "register split exceeds the launch allocation");
  static constexpr int A_ITEMS = CONV_A ? BM * 4 : 0;
  static constexpr int B_ITEMS = CONV_B ? BN * 4 : 0;
  static constexpr int ITEMS = A_ITEMS + B_ITEMS;
  static constexpr int IPT = ITEMS > 0 ? (ITEMS + CONV_THREADS - 1) / CONV_THREADS : 1;
  static constexpr int A8_BYTES = CONV_A ? BM * BK8 : 0;
  static constexpr int B8_BYTES = CONV_B ? BN * BK8 : 0;
  static constexpr int STAGE8 = A8_BYTES + B8_BYTES;
  static constexpr int A16_SUB = BM * BK16 * 2;           // one 64-K sub-tile of A
  static constexpr int B16_SUB = BN * BK16 * 2;
  static constexpr int A16_BYTES = A16_SUB * K64_PER_STAGE;
  static constexpr int B16_BYTES = B16_SUB * K64_PER_STAGE;
  static constexpr int STAGE16 = A16_BYTES + B16_BYTES;
  static constexpr int OFF_S8 = 0;
  static constexpr int OFF_S16 = OFF_S8 + (ANY_CONV ? S8 : 0) * STAGE8;
  static constexpr int OFF_EPI = OFF_S16 + S16 * STAGE16;   // 4 KB store staging per epilogue warp
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * 4096;
  // full8[S8] empty8[S8] full16[S16] tma16[S16] empty16[S16] pfull16[S16]
  // accfull[2] accempty[2] paccempty[2] done skstored skdecided sclfull sclfree
  // skload[EPI_WARPS]
  static constexpr int NUM_BARS = 2 * S8 + 4 * S16 + 11 + EPI_WARPS;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  // the current tile's per-channel scales (fp32) and bias (bf16), staged by
  // the epilogue warps: PAIR_N columns
  static constexpr int OFF_SCL = (OFF_MISC + 16 + 15) / 16 * 16;
  static constexpr int OFF_SCL_BIAS = OFF_SCL + PAIR_N * 4;
  static constexpr int SMEM_BYTES = OFF_SCL_BIAS + PAIR_N * 2 + 1024;
  static constexpr int TMEM_COLS = 2 * PAIR_N;
  // a stream-K finisher loads the other pairs' partials into the pipeline
  // buffers, 16 KB per epilogue warp
  static_assert(OFF_EPI >= EPI_WARPS * 16384, "stream-K partial buffers overlap the staging");
  static constexpr uint32_t TX8 = STAGE8;
  static constexpr uint32_t TX16 = (CONV_A ? 0 : A16_BYTES) + (CONV_B ? 0 : B16_BYTES);
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(STAGE8 % 1024 == 0 && STAGE16 % 1024 == 0, "stage alignment");
  static_assert(!WIDE || A16_SUB == B16_SUB, "wide stages: equal sub-tiles");
};

struct PairBars {
  uint32_t base;
  int S8, S16;
  __device__ uint32_t full8(int s) const { return base + 8u * s; }
  __device__ uint32_t empty8(int s) const { return base + 8u * (S8 + s); }
  __device__ uint32_t full16(int s) const { return base + 8u * (2 * S8 + s); }
  __device__ uint32_t tma16(int s) const { return base + 8u * (2 * S8 + S16 + s); }
  __device__ uint32_t empty16(int s) const { return base + 8u * (2 * S8 + 2 * S16 + s); }
  __device__ uint32_t pfull16(int s) const { return base + 8u * (2 * S8 + 3 * S16 + s); }
  __device__ uint32_t accfull(int b) const { return base + 8u * (2 * S8 + 4 * S16 + b); }
  __device__ uint32_t accempty(int b) const { return base + 8u * (2 * S8 + 4 * S16 + 2 + b); }
  __device__ uint32_t paccempty(int b) const { return base + 8u * (2 * S8 + 4 * S16 + 4 + b); }
  __device__ uint32_t done() const { return base + 8u * (2 * S8 + 4 * S16 + 6); }
  // stream-K fix-up: every epilogue warp's partial is stored / the decision
  // whether this CTA finishes the tile is made
  __device__ uint32_t skstored() const { return base + 8u * (2 * S8 + 4 * S16 + 7); }
  __device__ uint32_t skdecided() const { return base + 8u * (2 * S8 + 4 * S16 + 8); }
  // the staged per-channel scales: written (one arrive per epilogue warp) /
  // read by every epilogue warp
  __device__ uint32_t sclfull() const { return base + 8u * (2 * S8 + 4 * S16 + 9); }
  __device__ uint32_t sclfree() const { return base + 8u * (2 * S8 + 4 * S16 + 10); }
  // stream-K: epilogue warp w's TMA loads of the other pairs' partials
  __device__ uint32_t skload(int w) const { return base + 8u * (2 * S8 + 4 * S16 + 11 + w); }
};

struct PairTile {
  int mp, nb, ks, kb0, kb1;
  int tile;
  bool partial;      // stream-K: only part of the tile's K range
};

// Pair tiles: num_m_blk counts 256-row pair blocks, num_n_blk 256-column blocks.
__device__ __forceinline__ PairTile decode_pair_tile(const GemmParams& p, int tile) {
  PairTile t;
  t.ks = tile % p.splits;
  const int rest = tile / p.splits;
  tile_coords(p, rest, t.mp, t.nb);
  t.kb0 = t.ks * p.kb_per_split;
  t.kb1 = min(t.kb0 + p.kb_per_split, p.total_kb);
  return t;
}

// Stream-K: after sk_waves whole waves of tiles, the units of the remaining
// tiles are (tile, K-block) pairs in tile-major order, numbered from the
// first of those tiles; pair q of the Q = sk_pairs that share them owns
// units [sk_first(q), sk_first(q + 1)).  The host plans stream-K only when
// units * Q < 2^31, so 32-bit arithmetic is exact here.
__device__ __forceinline__ int sk_tile0(const GemmParams& p, int npairs) {
  return p.sk_waves * npairs;   // the first split-region tile
}
__device__ __forceinline__ uint32_t sk_units(const GemmParams& p, int npairs) {
  return static_cast<uint32_t>(p.num_tiles - sk_tile0(p, npairs)) * static_cast<uint32_t>(p.total_kb);
}
__device__ __forceinline__ uint32_t sk_first(const GemmParams& p, int q, int npairs) {
  return sk_units(p, npairs) * static_cast<uint32_t>(q) / static_cast<uint32_t>(p.sk_pairs);
}
// The pair whose range holds unit u: the largest q with sk_first(q) <= u.
__device__ __forceinline__ int sk_holder(const GemmParams& p, uint32_t u, int npairs) {
  return static_cast<int>(((u + 1) * static_cast<uint32_t>(p.sk_pairs) - 1) / sk_units(p, npairs));
}

// Item `it` of this pair's schedule; false once the pair has no more work.
// Without stream-K the items are the tiles pair, pair + P, ...; with it the
// first sk_waves items are those, and the rest the pieces of the pair's unit
// range cut at tile boundaries (only the first and the last piece can be
// part of a tile).
__device__ __forceinline__ bool pair_item(const GemmParams& p, int pair, int npairs, int it,
                                          PairTile& t) {
  if (!p.stream_k || it < p.sk_waves) {
    const int tile = pair + it * npairs;
    if (tile >= p.num_tiles) return false;
    t = decode_pair_tile(p, tile);
    t.tile = tile;
    t.partial = false;
    return true;
  }
  if (pair >= p.sk_pairs) return false;
  const uint32_t kb = static_cast<uint32_t>(p.total_kb);
  const uint32_t u0 = sk_first(p, pair, npairs);
  const uint32_t u1 = sk_first(p, pair + 1, npairs);
  const uint32_t rel = u0 / kb + static_cast<uint32_t>(it - p.sk_waves);   // tile within the region
  const uint32_t t0 = rel * kb;
  if (u0 >= u1 || t0 >= u1) return false;
  t.tile = sk_tile0(p, npairs) + static_cast<int>(rel);
  t.ks = 0;
  tile_coords(p, t.tile, t.mp, t.nb);
  t.kb0 = static_cast<int>((u0 > t0 ? u0 : t0) - t0);
  t.kb1 = static_cast<int>((u1 < t0 + kb ? u1 : t0 + kb) - t0);
  t.partial = t.kb0 > 0 || t.kb1 < p.total_kb;
  return true;
}

// Counts one arrival at a split tile's word and returns true for the n-th
// arrival of this launch.  A word left by an earlier launch carries another
// epoch and counts as zero, so the array never needs clearing.  Each
// failed exchange means another participant arrived, so the loop ends within
// n rounds; the bound only guards against a corrupted word.
__device__ __forceinline__ bool sk_arrive(unsigned long long* word, unsigned long long epoch,
                                          int n, bool& ok) {
  unsigned long long cur = atomicAdd(word, 0ull);
  for (int i = 0; i < 4096; ++i) {
    const unsigned long long cnt = (cur >> 16) == epoch ? (cur & 0xFFFFull) : 0ull;
    const unsigned long long prev = atomicCAS(word, cur, (epoch << 16) | (cnt + 1));
    if (prev == cur) return static_cast<int>(cnt + 1) == n;
    cur = prev;
  }
  ok = false;
  return false;
}

template <class Cfg>
__device__ __forceinline__ void pair_epilogue_role(const GemmParams& p, const CUtensorMap* tmY,
                                                   const CUtensorMap* tmP, uint32_t sbase,
                                                   uint32_t tmem_base, int warp, int lane,
                                                   uint32_t rank, volatile int* abort_flag,
                                                   volatile int* sk_flag, const PairBars& bars) {
  const int ew = warp - Cfg::EPI_WARP0;
  const int quarter = warp & 3;
  const int cg = ew >> 2;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const bool bf16_out = p.out_mode == kOutBf16;
  const uint32_t scl_w = sbase + Cfg::OFF_SCL;
  const uint32_t scl_b = sbase + Cfg::OFF_SCL_BIAS;
  Ring racc, rscl;
  bool ok = true;
  PairTile tc;
  for (int it = 0; ok && pair_item(p, pair, npairs, it, tc); ++it) {
    const int nst = 2 * (tc.kb1 - tc.kb0) / Cfg::K64_PER_STAGE;
    const int chunk = p.chunk_stages / Cfg::K64_PER_STAGE;
    const int m_loc = static_cast<int>(rank) * Cfg::BM + quarter * 32;  // rows within the tile
    const int n_loc = cg * 128;
    float sa = 0.0f;
    if (bf16_out) {
      // Stage this tile's per-channel scales and bias (once the previous
      // tile's readers are done with them) and load this lane's per-token
      // scale, while the tile's MMAs run: the loads' latency stays off the
      // path from the last accumulator to the store.
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.sclfree(), rscl.ph ^ 1u, abort_flag));
      if (!ok) break;
      stage_channel_scales(p, scl_w, scl_b, tc.nb * Cfg::PAIR_N, ew, lane);
      const int m = tc.mp * Cfg::PAIR_M + m_loc + lane;
      if (m < p.M) sa = p.s_a[m];
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.sclfull());
    }
    // Stream-K finisher (below): one thread checks, without waiting, at the
    // start of the piece whether every other piece's partial is already
    // published (the usual case: those pieces open their pairs' ranges), so
    // that the check's memory latency overlaps the MMAs; otherwise it waits
    // after the drains.  A drain is never held back by it.
    const bool sk_finisher = tc.partial && tc.kb0 == 0 && ew == 0 && lane == 0;
    bool sk_decided = false;
    auto sk_decide = [&](bool wait) {
      const uint32_t rel = static_cast<uint32_t>(tc.tile - sk_tile0(p, npairs));
      const int q0 = sk_holder(p, rel * static_cast<uint32_t>(p.total_kb), npairs);
      const int q1 = sk_holder(p, (rel + 1) * static_cast<uint32_t>(p.total_kb) - 1, npairs);
      unsigned long long* word = p.sk_arrive + 2 * tc.tile + rank;
      const unsigned long long want = (p.sk_epoch << 16) | static_cast<unsigned long long>(q1 - q0);
      bool fok;
      if (wait) {
        fok = gmem_wait_eq(word, want, abort_flag);   // bounded
      } else {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(word) : "memory");
        if (v != want) return;
        fok = true;
      }
      // the word is complete: clear it, which nothing else does in this
      // launch, so that a replay of the launch with the same epoch (a CUDA
      // graph) starts at zero
      if (fok) {
        *reinterpret_cast<volatile unsigned long long*>(word) = 0ull;
        fence_proxy_async_global();   // the partials are read by TMA below
      }
      *sk_flag = fok ? 1 : 0;
      mbar_arrive(bars.skdecided());   // always, so no epilogue warp waits in vain
      sk_decided = true;
    };
    int acc[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) acc[i] = 0;
    if (sk_finisher) sk_decide(false);
    for (int st0 = 0; st0 < nst; st0 += chunk) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.accfull(racc.s), racc.ph, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(racc.s * Cfg::PAIR_N + cg * 128);
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
      if (lane == 0) mbar_arrive(bars.accempty(racc.s));
      racc.advance(2);
    }
    if (!ok) break;
    if (bf16_out) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.sclfull(), rscl.ph, abort_flag));
      if (!ok) break;
    }
    const uint32_t stage = sbase + Cfg::OFF_EPI + static_cast<uint32_t>(ew) * 4096u;
    if (tc.partial) {
      // Stream-K fix-up.  The pair holding the tile's first K blocks (always
      // the last item of its range) finishes the tile; every other piece is
      // the first item of its pair's range, done early.  Those pairs publish
      // their int32 partials, each in its pair's slot (a pair publishes at
      // most once), and count themselves in the tile's arrival word.  The
      // finisher waits until the others have all arrived (above, while its
      // MMAs run), loads their partials by TMA into its own pipeline buffers
      // (idle once its last item's MMAs are done), adds them to the
      // accumulator it still holds and writes the tile.
      const uint32_t rel = static_cast<uint32_t>(tc.tile - sk_tile0(p, npairs));   // tile within the region
      const int q0 = sk_holder(p, rel * static_cast<uint32_t>(p.total_kb), npairs);
      const int q1 = sk_holder(p, (rel + 1) * static_cast<uint32_t>(p.total_kb) - 1, npairs);
      unsigned long long* word = p.sk_arrive + 2 * tc.tile + rank;
      if (tc.kb0 != 0) {
        store_warp_tile_s32<128>(tmP, stage, lane, m_loc, n_loc, acc, pair);
        if (lane == 0) {
          bulk_wait_all();             // the partial is in global memory
          fence_proxy_async_global();
          mbar_arrive(bars.skstored());
        }
        __syncwarp();
        if (ew == 0 && lane == 0) {
          // (a timed-out wait has raised the abort flag and the status word;
          // a pair publishes at most one partial, so the phase is 0)
          if (mbar_wait(bars.skstored(), 0u, abort_flag)) {
            bool aok = true;
            __threadfence();
            sk_arrive(word, p.sk_epoch, q1 - q0 + 1, aok);
            if (!aok) {
              *abort_flag = 1;
              atomicOr(&g_status, 1u << 5);  // I8_ERR_CUDA: corrupted arrival word
            }
          }
        }
      } else {
        if (sk_finisher && !sk_decided) sk_decide(true);
        // a pair finishes at most one tile, its last item: the phase is 0
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.skdecided(), 0u, abort_flag)) && *sk_flag != 0;
        if (!ok) break;
        // This warp's 32 rows x 128 columns of each other pair's slot: four
        // 32 x 32 int32 boxes (16 KB, 128-byte swizzle, the layout the
        // partial was stored with) into this warp's 16 KB of the buffers.
        const uint32_t buf = sbase + Cfg::OFF_S8 + static_cast<uint32_t>(ew) * 16384u;
        uint32_t lph = 0;
#pragma unroll 1
        for (int q = q0; ok && q <= q1; ++q) {
          if (q == pair) continue;
          if (lane == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bars.skload(ew), 16384u);
#pragma unroll
            for (int g = 0; g < 4; ++g)
              tma_load_3d(buf + 4096u * g, tmP, bars.skload(ew), n_loc + 32 * g, m_loc, q);
          }
          __syncwarp();
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.skload(ew), lph, abort_flag));
          lph ^= 1u;
          if (!ok) break;
          const uint32_t row = buf + static_cast<uint32_t>(lane) * 128u;
          const uint32_t x = static_cast<uint32_t>(lane & 7);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 v = lds128(row + 4096u * g + ((static_cast<uint32_t>(c) ^ x) << 4));
              acc[32 * g + 4 * c] += static_cast<int>(v.x);
              acc[32 * g + 4 * c + 1] += static_cast<int>(v.y);
              acc[32 * g + 4 * c + 2] += static_cast<int>(v.z);
              acc[32 * g + 4 * c + 3] += static_cast<int>(v.w);
            }
          }
          __syncwarp();   // every lane has read the boxes before the next load overwrites them
        }
        if (!ok) break;
        if (bf16_out)
          store_warp_tile_bf16_staged<128>(tmY, stage, lane, tc.mp * Cfg::PAIR_M + m_loc,
                                           tc.nb * Cfg::PAIR_N + n_loc, acc, sa, scl_w + 4u * n_loc,
                                           scl_b + 2u * n_loc);
        else
          store_warp_tile<128>(p, tmY, stage, lane, tc.mp * Cfg::PAIR_M + m_loc,
                               tc.nb * Cfg::PAIR_N + n_loc, acc, tc.ks);
      }
    } else if (bf16_out) {
      store_warp_tile_bf16_staged<128>(tmY, stage, lane, tc.mp * Cfg::PAIR_M + m_loc,
                                       tc.nb * Cfg::PAIR_N + n_loc, acc, sa, scl_w + 4u * n_loc,
                                       scl_b + 2u * n_loc);
    } else {
      store_warp_tile<128>(p, tmY, stage, lane, tc.mp * Cfg::PAIR_M + m_loc,
                           tc.nb * Cfg::PAIR_N + n_loc, acc, tc.ks);
    }
    if (bf16_out) {
      // this warp's reads of the staged scales are done
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.sclfree());
      rscl.advance(1);
    }
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

template <class Cfg>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg::THREADS, 1)
    gemm_w8a8_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmY,
                          const __grid_constant__ CUtensorMap tmP, const GemmParams p) {
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
  auto stage16 = [&](int s) { return sbase + Cfg::OFF_S16 + static_cast<uint32_t>(s * Cfg::STAGE16); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);
  volatile int* sk_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 8);

  if (warp >= 2 && lane == 0) {
    // The first read of a launch parameter misses the constant cache (about
    // 1 us on GB300) and would sit on every role's path to its first tile;
    // touch the fields the roles decode first while warps 0 and 1 set up the
    // barriers and the tensor memory.
    const int t = p.num_tiles ^ p.splits ^ p.total_kb ^ p.kb_per_split ^ p.num_m_blk ^
                  p.num_n_blk ^ p.n_fastest ^ p.stream_k ^ p.sk_waves ^ p.sk_pairs ^ p.chunk_stages ^
                  p.out_mode ^ p.M ^
                  p.N ^ static_cast<int>(reinterpret_cast<uintptr_t>(p.s_a)) ^
                  static_cast<int>(reinterpret_cast<uintptr_t>(p.s_w)) ^
                  static_cast<int>(reinterpret_cast<uintptr_t>(p.sk_arrive));
    asm volatile("" ::"r"(t));
    if constexpr (Cfg::ANY_CONV) {
      // The first int8 stages of this CTA's first item on their way into L2
      // while the previous kernel of the stream drains (prefetches cannot
      // leave stale data; the loads still wait for it).
      PairTile t0;
      if (warp == 2 && pair_item(p, pair, npairs, 0, t0)) {
        const int m0 = t0.mp * Cfg::PAIR_M + static_cast<int>(rank) * Cfg::BM;
        const int n0 = t0.nb * Cfg::PAIR_N + static_cast<int>(rank) * Cfg::BN;
        for (int kb = t0.kb0; kb < t0.kb1 && kb < t0.kb0 + Cfg::S8; ++kb) {
          if constexpr (Cfg::CONV_A) tma_prefetch_l2_2d(&tmA, kb * Cfg::BK8, m0);
          if constexpr (Cfg::CONV_B) tma_prefetch_l2_2d(&tmB, kb * Cfg::BK8, n0);
        }
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::S8; ++s) {
      mbar_init(bars.full8(s), 1);
      mbar_init(bars.empty8(s), Cfg::CONV_WARPS);
    }
    for (int s = 0; s < Cfg::S16; ++s) {
      mbar_init(bars.full16(s), Cfg::CONV_WARPS);
      mbar_init(bars.tma16(s), 1);
      mbar_init(bars.empty16(s), 1);
      mbar_init(bars.pfull16(s), 1);     // CTA 0: forwarded by CTA 1's relay
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.accfull(b), 1);
      mbar_init(bars.accempty(b), Cfg::EPI_WARPS);
      mbar_init(bars.paccempty(b), 1);   // CTA 0: forwarded by CTA 1's relay
    }
    mbar_init(bars.done(), 1);
    mbar_init(bars.skstored(), Cfg::EPI_WARPS);
    mbar_init(bars.skdecided(), 1);
    mbar_init(bars.sclfull(), Cfg::EPI_WARPS);
    mbar_init(bars.sclfree(), Cfg::EPI_WARPS);
    for (int w = 0; w < Cfg::EPI_WARPS; ++w) mbar_init(bars.skload(w), 1);
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
    if (p.stream_k) tma_prefetch_desc(&tmP);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // operands and outputs may belong to the previous kernel

  if (warp >= Cfg::EPI_WARP0) {
    regs_inc<Cfg::REG_HI>();
    pair_epilogue_role<Cfg>(p, &tmY, &tmP, sbase, tmem_base, warp, lane, rank, abort_flag,
                            sk_flag, bars);
  } else if (warp == 0) {
    regs_dec<Cfg::REG_LO>();
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Ring r8, r16;
      bool ok = true;
      PairTile tc;
      for (int it = 0; ok && pair_item(p, pair, npairs, it, tc); ++it) {
        const int m0 = tc.mp * Cfg::PAIR_M + static_cast<int>(rank) * Cfg::BM;
        const int n0 = tc.nb * Cfg::PAIR_N + static_cast<int>(rank) * Cfg::BN;
        for (int kb = tc.kb0; ok && kb < tc.kb1; ++kb) {
          if constexpr (Cfg::ANY_CONV) {
            if (!(ok = mbar_wait(bars.empty8(r8.s), r8.ph ^ 1u, abort_flag))) break;
            mbar_arrive_expect_tx(bars.full8(r8.s), Cfg::TX8);
            if constexpr (Cfg::CONV_A)
              tma_load_2d(stage8(r8.s), &tmA, bars.full8(r8.s), kb * Cfg::BK8, m0);
            if constexpr (Cfg::CONV_B)
              tma_load_2d(stage8(r8.s) + Cfg::A8_BYTES, &tmB, bars.full8(r8.s), kb * Cfg::BK8, n0);
            r8.advance(Cfg::S8);
          }
          if constexpr (Cfg::ANY_DIRECT) {
            // the fp16 operand: one stage per 64-K half, or (WIDE) both
            // halves as the two sub-tiles of one stage
            for (int h = 0; h < 2; h += Cfg::K64_PER_STAGE) {
              if (!(ok = mbar_wait(bars.empty16(r16.s), r16.ph ^ 1u, abort_flag))) break;
              mbar_arrive_expect_tx(bars.tma16(r16.s), Cfg::TX16);
#pragma unroll
              for (int q = 0; q < Cfg::K64_PER_STAGE; ++q) {
                const int k16 = kb * Cfg::BK8 + (h + q) * Cfg::BK16;
                if constexpr (!Cfg::CONV_A)
                  tma_load_2d(stage16(r16.s) + q * Cfg::A16_SUB, &tmA, bars.tma16(r16.s), k16, m0);
                if constexpr (!Cfg::CONV_B)
                  tma_load_2d(stage16(r16.s) + Cfg::A16_BYTES + q * Cfg::B16_SUB, &tmB,
                              bars.tma16(r16.s), k16, n0);
              }
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
      PairTile tc;
      for (int it = 0; ok && pair_item(p, pair, npairs, it, tc); ++it) {
        const int nst = 2 * (tc.kb1 - tc.kb0) / Cfg::K64_PER_STAGE;
        const int chunk = p.chunk_stages / Cfg::K64_PER_STAGE;
        for (int st0 = 0; ok && st0 < nst; st0 += chunk) {
          const int st1 = min(nst, st0 + chunk);
          if (!(ok = mbar_wait(bars.accempty(racc.s), racc.ph ^ 1u, abort_flag))) break;
          if (!(ok = Cfg::SYNC == 0
                         ? mbar_wait_cluster(bars.paccempty(racc.s), racc.ph ^ 1u, abort_flag)
                         : mbar_wait(bars.paccempty(racc.s), racc.ph ^ 1u, abort_flag)))
            break;
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(racc.s * Cfg::PAIR_N);
          for (int st = st0; st < st1; ++st) {
            if (!(ok = mbar_wait(bars.full16(r16.s), r16.ph, abort_flag))) break;
            if (!(ok = Cfg::SYNC == 0 ? mbar_wait_cluster(bars.pfull16(r16.s), r16.ph, abort_flag)
                                      : mbar_wait(bars.pfull16(r16.s), r16.ph, abort_flag)))
              break;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < Cfg::K64_PER_STAGE; ++h) {
              const uint64_t ad = smem_desc_sw128(stage16(r16.s) + h * Cfg::A16_SUB);
              const uint64_t bd = smem_desc_sw128(stage16(r16.s) + Cfg::A16_BYTES + h * Cfg::B16_SUB);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                mma_f16_ss_pair(d, ad + 2u * j, bd + 2u * j, idesc,
                                (st > st0 || h > 0 || j > 0) ? 1u : 0u);
              }
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
      // Walks the MMA thread's schedule and forwards each completed phase of
      // this CTA's full16 / accempty barriers to CTA 0.  The first use of
      // each accumulator buffer needs no drain, so nothing is forwarded then.
      const uint32_t pfull0 = mapa_shared(bars.pfull16(0), 0);
      const uint32_t pacc0 = mapa_shared(bars.paccempty(0), 0);
      Ring r16, racc;
      int chunk = 0;
      bool ok = true;
      PairTile tc;
      for (int it = 0; ok && pair_item(p, pair, npairs, it, tc); ++it) {
        const int nst = 2 * (tc.kb1 - tc.kb0) / Cfg::K64_PER_STAGE;
        const int cst = p.chunk_stages / Cfg::K64_PER_STAGE;
        for (int st0 = 0; ok && st0 < nst; st0 += cst, ++chunk) {
          const int st1 = min(nst, st0 + cst);
          if (chunk >= 2) {
            if (!(ok = mbar_wait(bars.accempty(racc.s), racc.ph ^ 1u, abort_flag))) break;
            if constexpr (Cfg::SYNC == 2) mbar_arrive_remote_cta(pacc0 + 8u * racc.s);
            else mbar_arrive_cluster(pacc0 + 8u * racc.s);
          }
          racc.advance(2);
          for (int st = st0; st < st1; ++st) {
            if (!(ok = mbar_wait(bars.full16(r16.s), r16.ph, abort_flag))) break;
            if constexpr (Cfg::SYNC == 2) mbar_arrive_remote_cta(pfull0 + 8u * r16.s);
            else mbar_arrive_cluster(pfull0 + 8u * r16.s);
            r16.advance(Cfg::S16);
          }
        }
      }
    }
  } else {
    regs_dec<Cfg::REG_LO>();
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - 64;
    ConvItem items[Cfg::IPT];
#pragma unroll
    for (int j = 0; j < Cfg::IPT; ++j) {
      const int i = ct + j * Cfg::CONV_THREADS;
      items[j] = conv_item<Cfg>(i < Cfg::ITEMS ? i : 0);
    }
    Ring r8, r16;
    bool ok = true;
    PairTile tc;
    for (int it = 0; ok && pair_item(p, pair, npairs, it, tc); ++it) {
      for (int kb = tc.kb0; kb < tc.kb1; ++kb) {
        // Both K-halves of the int8 block are read from shared memory in one
        // batch, so the load latency is exposed once per block.
        uint4 v[2][Cfg::IPT];
        if constexpr (Cfg::ANY_CONV) {
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.full8(r8.s), r8.ph, abort_flag));
          if (!ok) break;
          const uint32_t s8 = stage8(r8.s);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < Cfg::IPT; ++j) {
              if (ct + j * Cfg::CONV_THREADS < Cfg::ITEMS)
                v[h][j] = lds128(s8 + (items[j].src ^ (static_cast<uint32_t>(h) << 6)));
            }
          }
        }
        if constexpr (Cfg::WIDE) {
          // both K-halves into the two sub-tiles of one fp16 stage
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.empty16(r16.s), r16.ph ^ 1u, abort_flag));
          if (!ok) break;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t s16 = stage16(r16.s) + static_cast<uint32_t>(h * Cfg::A16_SUB);
#pragma unroll
            for (int j = 0; j < Cfg::IPT; ++j) {
              if (ct + j * Cfg::CONV_THREADS < Cfg::ITEMS) {
                uint4 o0, o1;
                s8x4_to_f16x4(v[h][j].x, o0.x, o0.y);
                s8x4_to_f16x4(v[h][j].y, o0.z, o0.w);
                s8x4_to_f16x4(v[h][j].z, o1.x, o1.y);
                s8x4_to_f16x4(v[h][j].w, o1.z, o1.w);
                sts128(s16 + items[j].dst, o0);
                sts128(s16 + (items[j].dst ^ 16u), o1);
              }
            }
          }
          fence_proxy_async_smem();
          if constexpr (Cfg::ANY_DIRECT) {
            // this CTA's directly loaded operand of the stage must have landed
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.tma16(r16.s), r16.ph, abort_flag));
            if (!ok) break;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.full16(r16.s));
          r16.advance(Cfg::S16);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.empty16(r16.s), r16.ph ^ 1u, abort_flag));
            if (!ok) break;
            if constexpr (Cfg::ANY_CONV) {
              const uint32_t s16 = stage16(r16.s);
#pragma unroll
              for (int j = 0; j < Cfg::IPT; ++j) {
                if (ct + j * Cfg::CONV_THREADS < Cfg::ITEMS) {
                  uint4 o0, o1;
                  s8x4_to_f16x4(v[h][j].x, o0.x, o0.y);
                  s8x4_to_f16x4(v[h][j].y, o0.z, o0.w);
                  s8x4_to_f16x4(v[h][j].z, o1.x, o1.y);
                  s8x4_to_f16x4(v[h][j].w, o1.z, o1.w);
                  sts128(s16 + items[j].dst, o0);
                  sts128(s16 + (items[j].dst ^ 16u), o1);
                }
              }
              fence_proxy_async_smem();
            }
            if constexpr (Cfg::ANY_DIRECT) {
              // this CTA's directly loaded half of the stage must have landed
              ok = __all_sync(0xFFFFFFFFu, mbar_wait(bars.tma16(r16.s), r16.ph, abort_flag));
              if (!ok) break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.full16(r16.s));
            r16.advance(Cfg::S16);
          }
        }
        if (!ok) break;
        if constexpr (Cfg::ANY_CONV) {
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.empty8(r8.s));
          r8.advance(Cfg::S8);
        }
      }
    }
  }

  __syncwarp();
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's MMAs and remote arrivals are finished
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace i8
