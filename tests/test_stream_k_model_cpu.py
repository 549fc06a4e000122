"""The stream-K schedule of the CTA-pair GEMM, modelled on the CPU.

Stream-K splits the (tile, K-block) units of a GEMM evenly over the P CTA
pairs of a persistent launch; tiles cut between pairs are finished by the
last pair to arrive, from every participant's exact int32 partial.  The
schedule is integer arithmetic only, so it can be checked here for many
shapes.  The model restates the kernel's formulas:
  units U = tiles * kb (tile-major), pair q owns [first(q), first(q + 1))
  with first(q) = U * q // P; its item `it` is tile first(q) // kb + it,
  cut to the pair's range; holder(u) = ((u + 1) * P - 1) // U;
  a split tile's participants are holder(first unit) .. holder(last unit);
  a partial piece is stored in slot 2q + (it == 0 ? 0 : 1) and read back from
  slot 2q + (first(q) // kb == tile ? 0 : 1); the fix-up barriers of a pair
  are in phase (it > 0 and first(q) % kb != 0).
and checks what correctness needs: every unit computed once, every tile's K
blocks covered once, at most two split pieces per pair (its first and its
last), consistent slots, arrival counts and barrier phases.  The host plans
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
                for idx, it in enumerate(partial_its):
                    # the fix-up barriers' phase: how many split pieces came before
                    phase = 1 if (it > 0 and first(U, q, P) % kb != 0) else 0
                    assert phase == idx % 2, (tiles, kb, P, q)
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
                # each participant's partial is read from the slot it stored
                for q, it, _, _ in ps:
                    store = 2 * q + (0 if it == 0 else 1)
                    read = 2 * q + (0 if first(U, q, P) // kb == tile else 1)
                    assert store == read
            # no slot is written twice
            used = [2 * q + (0 if it == 0 else 1)
                    for ps in pieces.values() if len(ps) > 1 for q, it, _, _ in ps]
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
        "2 * pair + (it == 0 ? 0 : 1)",
        "2 * q + (sk_first(p, q, npairs) / static_cast<uint32_t>(p.total_kb) == "
        "static_cast<uint32_t>(tc.tile) ? 0 : 1);",
        "(it > 0 && sk_first(p, pair, npairs) % static_cast<uint32_t>(p.total_kb) != 0) ? 1u : 0u;",
        "last_pair() - first_pair() + 1",
    ]:
        assert " ".join(text.split()) in src, text
