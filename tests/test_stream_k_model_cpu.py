"""The stream-K schedule of the CTA-pair GEMM, modelled on the CPU.

Stream-K splits the (tile, K-block) units of a GEMM evenly over the P CTA
pairs of a persistent launch.  A tile cut between pairs is finished by the
pair holding its first K blocks, from the accumulator it still holds plus the
exact int32 partials the other participants published.  The schedule is
integer arithmetic only, so it can be checked here for many shapes.  The
model restates the kernel's formulas:
  units U = tiles * kb (tile-major), pair q owns [first(q), first(q + 1))
  with first(q) = U * q // P; its item `it` is tile first(q) // kb + it,
  cut to the pair's range; holder(u) = ((u + 1) * P - 1) // U;
  a split tile's participants are holder(first unit) .. holder(last unit);
  the piece starting at K block 0 finishes the tile, every other piece
  publishes its partial in its pair's slot q, which the finisher reads back;
  the finisher waits for the other participants' q1 - q0 arrivals; every
  fix-up barrier is used in phase 0.
and checks what correctness needs: every unit computed once, every tile's K
blocks covered once, at most two split pieces per pair (its first and its
last), the finisher's piece the last item of its pair and every published
piece the first item of its pair (so a pair publishes at most once, which
one slot per pair needs, and finishes at most once, which phase 0 needs),
and a finisher never
waiting on a pair below it (the waits cannot form a cycle).  The host plans
P = min(resident pairs, max(1, U // 4)), so every pair owns at least one unit
(at least four whenever U >= 4).
"""
import pytest

TILES = [1, 2, 3, 5, 8, 13, 36, 74, 75, 100, 148, 149, 360, 500]
KBS = [1, 4, 5, 8, 24, 31, 64, 96, 128, 1024]
SLOTS = [1, 2, 37, 74, 76, 148]


def first(U, q, P):
    return U * q // P


def holder(U, u, P):
    return ((u + 1) * P - 1) // U


def pair_items(U, kb, q, P):
    """The pieces (it, tile, kb0, kb1) of pair q, as the kernel walks them."""
    u0, u1 = first(U, q, P), first(U, q + 1, P)
    out = []
    it = 0
    while True:
        tile = u0 // kb + it
        t0 = tile * kb
        if u0 >= u1 or t0 >= u1:
            return out
        out.append((it, tile, max(u0, t0) - t0, min(u1, t0 + kb) - t0))
        it += 1


@pytest.mark.parametrize("tiles", TILES)
def test_stream_k_schedule(tiles):
    for kb in KBS:
        for slots in SLOTS:
            U = tiles * kb
            P = min(slots, max(1, U // 4))
            assert U * P < 2 ** 31                      # the kernel's 32-bit arithmetic
            # the ranges partition the units; none is empty
            bounds = [first(U, q, P) for q in range(P + 1)]
            assert bounds[0] == 0 and bounds[-1] == U
            assert all(b < c for b, c in zip(bounds, bounds[1:]))
            if U >= 4:
                assert all(c - b >= 4 for b, c in zip(bounds, bounds[1:]))
            # holder(u) is the pair whose range holds u
            for u in sorted({0, U - 1, *bounds[1:-1], *(b - 1 for b in bounds[1:-1])}):
                q = holder(U, u, P)
                assert bounds[q] <= u < bounds[q + 1], (tiles, kb, P, u)
            pieces = {}                                 # tile -> [(q, it, kb0, kb1)]
            for q in range(P):
                items = pair_items(U, kb, q, P)
                partial_its = [it for it, _, k0, k1 in items if k0 > 0 or k1 < kb]
                # split pieces only at a pair's first and last item
                assert all(it in (0, len(items) - 1) for it in partial_its)
                assert len(partial_its) <= 2
                # a pair publishes at most one piece (its first) and finishes
                # at most one (its last): each fix-up barrier is used once, in
                # phase 0
                publish = [it for it, _, k0, k1 in items if k0 > 0]
                finish = [it for it, _, k0, k1 in items if k0 == 0 and k1 < kb]
                assert publish in ([], [0]), (tiles, kb, P, q)
                assert finish in ([], [len(items) - 1]), (tiles, kb, P, q)
                for it, tile, k0, k1 in items:
                    assert 0 <= k0 < k1 <= kb
                    pieces.setdefault(tile, []).append((q, it, k0, k1))
            assert sorted(pieces) == list(range(tiles))
            for tile, ps in pieces.items():
                # the tile's K blocks covered once, in pair order
                ps.sort()
                assert ps[0][2] == 0 and ps[-1][3] == kb
                assert all(a[3] == b[2] for a, b in zip(ps, ps[1:]))
                split = len(ps) > 1
                assert split == any(k0 > 0 or k1 < kb for _, _, k0, k1 in ps)
                if not split:
                    continue
                # participants: holder of the first unit .. holder of the last
                q0 = holder(U, tile * kb, P)
                q1 = holder(U, (tile + 1) * kb - 1, P)
                assert [q for q, *_ in ps] == list(range(q0, q1 + 1))
                # the finisher is the first participant; the others publish,
                # so it waits for q1 - q0 arrivals from pairs above it
                fin = [q for q, it, k0, _ in ps if k0 == 0]
                assert fin == [q0]
                pubs = [(q, it) for q, it, k0, _ in ps if k0 > 0]
                assert len(pubs) == q1 - q0 and all(q > q0 for q, _ in pubs)
            # no slot (one per pair) is written twice
            used = [q for ps in pieces.values() if len(ps) > 1 for q, it, k0, _ in ps if k0 > 0]
            assert len(used) == len(set(used))


def test_model_restates_the_kernel_source():
    """The formulas above are the kernel's: if the kernel changes them, this
    fails and the model must be brought up to date."""
    import os
    src_path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "w8a8_int8_quantized_i8_gb300", "csrc", "gemm_pair.cuh")
    with open(src_path) as fh:
        src = " ".join(fh.read().split())
    for text in [
        "return static_cast<uint32_t>(p.num_tiles) * static_cast<uint32_t>(p.total_kb);",
        "return sk_units(p) * static_cast<uint32_t>(q) / static_cast<uint32_t>(npairs);",
        "return static_cast<int>(((u + 1) * static_cast<uint32_t>(npairs) - 1) / sk_units(p));",
        "const uint32_t tile = u0 / kb + static_cast<uint32_t>(it);",
        "if (u0 >= u1 || t0 >= u1) return false;",
        "t.kb0 = static_cast<int>((u0 > t0 ? u0 : t0) - t0);",
        "t.kb1 = static_cast<int>((u1 < t0 + kb ? u1 : t0 + kb) - t0);",
        "store_warp_tile_s32<128>(tmP, stage, lane, m_loc, n_loc, acc, pair);",
        "tma_load_3d(buf + 4096u * g, tmP, bars.skload(ew), n_loc + 32 * g, m_loc, q);",
        "if (tc.kb0 != 0) {",
        "sk_arrive(word, p.sk_epoch, q1 - q0 + 1, aok);",
        "gmem_wait_eq(word, (p.sk_epoch << 16) | static_cast<unsigned long long>(q1 - q0),",
        "mbar_wait(bars.skstored(), 0u, abort_flag)",
        "mbar_wait(bars.skdecided(), 0u, abort_flag)",
        "if (q == pair) continue;",
    ]:
        assert " ".join(text.split()) in src, text
