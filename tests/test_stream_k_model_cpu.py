"""The stream-K schedule of the CTA-pair GEMM, modelled on the CPU.

The P CTA pairs of a persistent launch first take W whole waves of tiles
(tile = pair + wave * P, neighbouring tiles in flight together); the units
(tile, K block) of the remaining tiles are then split evenly over the first Q
pairs.  A tile cut between pairs is finished by the pair holding its first K
blocks, from the accumulator it still holds plus the exact int32 partials the
other participants published.  The schedule is integer arithmetic only, so it
can be checked here for many shapes.  The model restates the kernel's
formulas:
  the split region starts at tile W * P; its units U = (tiles - W * P) * kb
  are numbered tile-major from there; pair q < Q owns [first(q), first(q + 1))
  with first(q) = U * q // Q; its item W + j is region tile first(q) // kb + j,
  cut to the pair's range; holder(u) = ((u + 1) * Q - 1) // U;
  a split tile's participants are holder(first unit) .. holder(last unit);
  the piece starting at K block 0 finishes the tile, every other piece
  publishes its partial in its pair's slot q, which the finisher reads back;
  the finisher waits for the other participants' q1 - q0 arrivals; every
  fix-up barrier is used in phase 0.
and checks what correctness needs: every unit computed once, every tile's K
blocks covered once, at most two split pieces per pair (its first and its
last split-region item), the finisher's piece the last item of its pair and
every published piece the first split-region item of its pair (so a pair
publishes at most once, which one slot per pair needs, and finishes at most
once, which phase 0 needs), and a finisher never waiting on a pair below it
(the waits cannot form a cycle).  For K blocks >= 64 the host plans W =
tiles // P with every resident pair launched, else W = 0 with P =
min(resident pairs, max(1, U // 4)); Q = min(P, max(1, U // 4)).
"""
import pytest

import w8a8_int8_quantized_i8_gb300 as i8

TILES = [1, 2, 3, 5, 8, 13, 36, 74, 75, 100, 148, 149, 360, 500]
KBS = [1, 4, 5, 8, 24, 31, 64, 96, 128, 1024]
SLOTS = [1, 2, 37, 74, 76, 148]


def plan(tiles, kb, slots):
    """(P, W, Q) as the host plans them."""
    W = tiles // slots if kb >= 64 else 0
    P = slots if W > 0 else min(slots, max(1, tiles * kb // 4))
    U = (tiles - W * P) * kb
    Q = min(P, max(1, U // 4))
    return P, W, Q


def pair_items(tiles, kb, P, W, Q, q):
    """The items (it, tile, kb0, kb1) of pair q, as the kernel walks them."""
    out = []
    for it in range(W):
        tile = q + it * P
        if tile < tiles:
            out.append((it, tile, 0, kb))
    if q >= Q:
        return out
    U = (tiles - W * P) * kb
    u0, u1 = U * q // Q, U * (q + 1) // Q
    j = 0
    while True:
        rel = u0 // kb + j
        t0 = rel * kb
        if u0 >= u1 or t0 >= u1:
            return out
        out.append((W + j, W * P + rel, max(u0, t0) - t0, min(u1, t0 + kb) - t0))
        j += 1


def check(tiles, kb, P, W, Q):
    U = (tiles - W * P) * kb
    assert U > 0 and U * Q < 2 ** 31                 # the kernel's 32-bit arithmetic
    first = lambda q: U * q // Q                     # noqa: E731
    holder = lambda u: ((u + 1) * Q - 1) // U        # noqa: E731
    bounds = [first(q) for q in range(Q + 1)]
    assert bounds[0] == 0 and bounds[-1] == U
    assert all(b < c for b, c in zip(bounds, bounds[1:]))      # no empty range
    for u in sorted({0, U - 1, *bounds[1:-1], *(b - 1 for b in bounds[1:-1])}):
        q = holder(u)
        assert bounds[q] <= u < bounds[q + 1], (tiles, kb, P, W, Q, u)
    pieces = {}                                     # tile -> [(q, it, kb0, kb1)]
    for q in range(P):
        items = pair_items(tiles, kb, P, W, Q, q)
        split = [(it, k0, k1) for it, _, k0, k1 in items if k0 > 0 or k1 < kb]
        publish = [it for it, k0, _ in split if k0 > 0]
        finish = [it for it, k0, k1 in split if k0 == 0]
        # a pair publishes at most once (its first split-region item) and
        # finishes at most once (its last item): each fix-up barrier is used
        # once, in phase 0, and one slot per pair suffices
        assert publish in ([], [W]), (tiles, kb, P, W, Q, q)
        assert finish in ([], [len(items) - 1]), (tiles, kb, P, W, Q, q)
        for it, tile, k0, k1 in items:
            assert 0 <= k0 < k1 <= kb
            pieces.setdefault(tile, []).append((q, it, k0, k1))
    assert sorted(pieces) == list(range(tiles))
    for tile, ps in pieces.items():
        ps.sort()
        assert ps[0][2] == 0 and ps[-1][3] == kb
        assert all(a[3] == b[2] for a, b in zip(ps, ps[1:]))
        if len(ps) == 1:
            continue
        assert tile >= W * P                         # only the split region is cut
        rel = tile - W * P
        q0, q1 = holder(rel * kb), holder((rel + 1) * kb - 1)
        assert [q for q, *_ in ps] == list(range(q0, q1 + 1))
        # the finisher is the first participant; the others publish, so it
        # waits for q1 - q0 arrivals from pairs above it
        assert [q for q, _, k0, _ in ps if k0 == 0] == [q0]
        pubs = [q for q, _, k0, _ in ps if k0 > 0]
        assert len(pubs) == q1 - q0 and all(q > q0 for q in pubs)
    used = [q for ps in pieces.values() if len(ps) > 1 for q, _, k0, _ in ps if k0 > 0]
    assert len(used) == len(set(used))


@pytest.mark.parametrize("tiles", TILES)
def test_stream_k_schedule(tiles):
    for kb in KBS:
        for slots in SLOTS:
            if tiles % slots == 0:
                continue                             # the host never plans stream-K then
            check(tiles, kb, *plan(tiles, kb, slots))


def test_stream_k_schedule_of_the_host_plans():
    """The same checks on the host planner's own plans (forced stream-K)."""
    i8.set_option("stream_k", 2)
    n = 0
    try:
        for M in (256, 512, 1024, 2560, 4096, 8704):
            for N in (256, 768, 3072, 9216, 12288):
                for K in (128, 640, 3072, 12288):
                    p = i8.plan_query(M, N, K, "int8", sms=152, pairs=76, skinny_slots=304)
                    if p["kernel"] != "pair_stream_k":
                        continue
                    tiles, P = p["num_m"] * p["num_n"], p["grid"] // 2
                    assert (P, p["sk_waves"], p["sk_pairs"]) == plan(tiles, p["total_kb"], 76)
                    check(tiles, p["total_kb"], P, p["sk_waves"], p["sk_pairs"])
                    n += 1
    finally:
        i8.set_option("stream_k", 1)
    assert n > 50


def test_model_restates_the_kernel_source():
    """The formulas above are the kernel's: if the kernel changes them, this
    fails and the model must be brought up to date."""
    import os
    src_path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "w8a8_int8_quantized_i8_gb300", "csrc", "gemm_pair.cuh")
    with open(src_path) as fh:
        src = " ".join(fh.read().split())
    for text in [
        "return p.sk_waves * npairs;",
        "return static_cast<uint32_t>(p.num_tiles - sk_tile0(p, npairs)) * static_cast<uint32_t>(p.total_kb);",
        "return sk_units(p, npairs) * static_cast<uint32_t>(q) / static_cast<uint32_t>(p.sk_pairs);",
        "return static_cast<int>(((u + 1) * static_cast<uint32_t>(p.sk_pairs) - 1) / sk_units(p, npairs));",
        "if (!p.stream_k || it < p.sk_waves) { const int tile = pair + it * npairs;",
        "if (pair >= p.sk_pairs) return false;",
        "const uint32_t rel = u0 / kb + static_cast<uint32_t>(it - p.sk_waves);",
        "if (u0 >= u1 || t0 >= u1) return false;",
        "t.tile = sk_tile0(p, npairs) + static_cast<int>(rel);",
        "t.kb0 = static_cast<int>((u0 > t0 ? u0 : t0) - t0);",
        "t.kb1 = static_cast<int>((u1 < t0 + kb ? u1 : t0 + kb) - t0);",
        "const int q0 = sk_holder(p, rel * static_cast<uint32_t>(p.total_kb), npairs);",
        "const int q1 = sk_holder(p, (rel + 1) * static_cast<uint32_t>(p.total_kb) - 1, npairs);",
        "if (tc.kb0 != 0) {",
        "sk_arrive(word, p.sk_epoch, q1 - q0 + 1, aok);",
        "const unsigned long long want = (p.sk_epoch << 16) | static_cast<unsigned long long>(q1 - q0);",
        "fok = gmem_wait_eq(word, want, abort_flag);",
        "mbar_wait(bars.skstored(), 0u, abort_flag)",
        "mbar_wait(bars.skdecided(), 0u, abort_flag)",
        "if (q == pair) continue;",
        "store_warp_tile_s32<128>(tmP, stage, lane, m_loc, n_loc, acc, pair);",
        "tma_load_3d(buf + 4096u * g, tmP, bars.skload(ew), n_loc + 32 * g, m_loc, q);",
    ]:
        assert " ".join(text.split()) in src, text
