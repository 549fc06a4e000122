"""The tiled kernels' work decode, modelled on the CPU against the real plans.

Every tiled GEMM kernel (single CTA, CTA pair, direct) walks work items
item = worker + it * workers and decodes each as: split ks = item % splits,
output tile = item / splits, tile -> (m block, n block) by the tile order
(N blocks fastest or M blocks fastest), K blocks [ks * kb_per_split,
min((ks + 1) * kb_per_split, total_kb)).  Here that decode, restated, is fed
the plans the library's own host planner makes (i8_plan_query, no GPU) for
every route over a grid of shapes, and the test checks that the items cover
every output tile once per split, that each tile's splits partition its K
blocks with none empty, and that the tile order is a bijection.  A last test
ties the restated decode to the kernel sources.
"""
import os

import pytest

from w8a8_int8_quantized_i8_gb300 import binding as i8

GB300 = dict(sms=152, pairs=74, skinny_slots=304)
MS = [1, 9, 100, 255, 256, 300, 1024, 2560, 4352, 8704]
NS = [16, 200, 768, 3072, 9216]
KS = [16, 512, 3072, 12288, 131072]


def tile_coords(n_fastest, tile, num_m, num_n):
    if n_fastest:
        return tile // num_n, tile % num_n
    return tile % num_m, tile // num_m


def decode(item, splits, kb_per_split, total_kb, n_fastest, num_m, num_n):
    ks = item % splits
    mb, nb = tile_coords(n_fastest, item // splits, num_m, num_n)
    kb0 = ks * kb_per_split
    return mb, nb, ks, kb0, min(kb0 + kb_per_split, total_kb)


@pytest.mark.parametrize("route", ["int8", "w16", "f16codes", "e4m3"])
def test_items_cover_every_tile_and_k_block_once(route):
    checked = 0
    for M in MS:
        for N in NS:
            for K in KS:
                p = i8.plan_query(M, N, K, route, **GB300)
                if p["kernel"] in ("skinny", "pair_stream_k"):
                    continue
                nm, nn, s = p["num_m"], p["num_n"], p["splits"]
                items = nm * nn * s
                workers = p["grid"] // 2 if p["kernel"] in ("pair", "direct") else p["grid"]
                seen = {}
                for w in range(workers):
                    for item in range(w, items, workers):     # the persistent loop
                        mb, nb, ks, kb0, kb1 = decode(item, s, p["kb_per_split"], p["total_kb"],
                                                      p["n_fastest"], nm, nn)
                        assert 0 <= mb < nm and 0 <= nb < nn
                        assert 0 <= kb0 < kb1 <= p["total_kb"], (route, M, N, K, item)
                        assert (mb, nb, ks) not in seen
                        seen[(mb, nb, ks)] = (kb0, kb1)
                assert len(seen) == items
                for mb in range(nm):
                    for nb in range(nn):
                        ranges = sorted(seen[(mb, nb, ks)] for ks in range(s))
                        assert ranges[0][0] == 0 and ranges[-1][1] == p["total_kb"]
                        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
                checked += 1
    assert checked > 100


@pytest.mark.parametrize("num_m,num_n", [(1, 1), (1, 36), (34, 12), (10, 36), (7, 3)])
def test_tile_order_is_a_bijection_in_both_orders(num_m, num_n):
    for n_fastest in (0, 1):
        got = [tile_coords(n_fastest, t, num_m, num_n) for t in range(num_m * num_n)]
        assert sorted(got) == [(m, n) for m in range(num_m) for n in range(num_n)]
        # consecutive tiles share the operand the order keeps in L2
        if num_m > 1 and num_n > 1:
            a, b = got[0], got[1]
            assert (a[0] == b[0]) if n_fastest else (a[1] == b[1])


def test_model_restates_the_kernel_sources():
    root = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "w8a8_int8_quantized_i8_gb300", "csrc")

    def text(name):
        with open(os.path.join(root, name)) as fh:
            return " ".join(fh.read().split())

    order = ("if (p.n_fastest) { nb = tile % p.num_n_blk; mb = tile / p.num_n_blk; } "
             "else { mb = tile % p.num_m_blk; nb = tile / p.num_m_blk; }")
    assert order in text("gemm.cuh")
    for name, idx, rest, coords in [("gemm.cuh", "tile", "rest", "t.mb, t.nb"),
                                    ("gemm_pair.cuh", "tile", "rest", "t.mp, t.nb"),
                                    ("gemm_direct.cuh", "item", "tile", "t.mp, t.nb")]:
        body = (f"t.ks = {idx} % p.splits; const int {rest} = {idx} / p.splits; "
                f"tile_coords(p, {rest}, {coords}); t.kb0 = t.ks * p.kb_per_split; "
                f"t.kb1 = min(t.kb0 + p.kb_per_split, p.total_kb);")
        assert body in text(name), name


def test_skinny_splits_partition_the_k_stages():
    """The weight-streaming kernel: CTA x streams 64 weight rows of N-block
    x / S over the 256-K stages [r * ks_per_cta, min((r + 1) * ks_per_cta,
    num_ks)) of split r = x % S, its rank in the N-block's cluster of S CTAs;
    rank r owns outputs [cut(r), cut(r + 1)) of the block's E, cut(r) =
    E r / S, and the other ranks add their partials of those into r's."""
    n = 0
    for M in (1, 2, 3, 8):
        for N in (16, 200, 768, 3072, 9216, 18432):
            for K in (16, 512, 528, 3072, 12288, 131072):
                p = i8.plan_query(M, N, K, "int8", **GB300)
                if p["kernel"] != "skinny":
                    continue
                s, per, nks = p["splits"], p["kb_per_split"], p["total_kb"]
                assert nks == -(-K // 256) and p["num_n"] == -(-N // 64)
                assert 1 <= s <= 8 and p["grid"] == p["num_n"] * s
                ranges = [(r * per, min(r * per + per, nks)) for r in range(s)]
                assert all(a < b for a, b in ranges)
                assert ranges[0][0] == 0 and ranges[-1][1] == nks
                assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
                # every CTA of the grid: one N-block, one split, each pair once
                cover = {(x // s, x % s) for x in range(p["grid"])}
                assert len(cover) == p["grid"] and {b for b, _ in cover} == set(range(p["num_n"]))
                # the owned slices partition the block's outputs, none empty
                E = min(M, 8) * 64
                cut = [E * r // s for r in range(s + 1)]
                assert cut[0] == 0 and cut[-1] == E
                assert all(a < b for a, b in zip(cut, cut[1:]))
                # the owner search finds the slice of every output
                for e in range(E):
                    r = max([0] + [rr for rr in range(1, s) if cut[rr] <= e])
                    assert cut[r] <= e < cut[r + 1]
                n += 1
    assert n > 50
    src_path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "w8a8_int8_quantized_i8_gb300", "csrc", "skinny.cuh")
    with open(src_path) as fh:
        src = " ".join(fh.read().split())
    for text in ["const int split = static_cast<int>(blockIdx.x) % p.splits;",
                 "const int n0 = (static_cast<int>(blockIdx.x) / p.splits) * kSkinnyRows;",
                 "const int ks0 = split * p.ks_per_cta;",
                 "const int ks1 = min(ks0 + p.ks_per_cta, p.num_ks);",
                 "auto cut = [&](int r) { return E * r / S; };",
                 "const int own0 = cut(split);",
                 "const int own1 = cut(split + 1);",
                 "for (int rr = 1; rr < S; ++rr) if (cut(rr) <= e) r = rr;"]:
        assert text in src, text
