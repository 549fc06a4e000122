"""The shape -> configuration table (i8_plan_query), on the host.

The pages autotune their Triton kernel per shape ("Realizing Native INT8
Compute for Diffusion Transformers on Consumer GPUs", abstract); the library
instead picks tiles, split counts, schedules and tile order from a fixed
table.  These tests run that table for hand-described machines (no GPU) and
check what must hold for every plan -- every output tile and every K block
covered exactly once, no empty split, a grid that fits the machine, the
workspace the partials need -- plus each rule of the table and each option.
"""
import ctypes
import math

import pytest
import torch

from w8a8_int8_quantized_i8_gb300 import binding as i8

GB300 = dict(sms=152, pairs=74, skinny_slots=304)
MACHINES = [GB300, dict(sms=152, pairs=0, skinny_slots=0), dict(sms=20, pairs=9, skinny_slots=40)]
ROUTES = ["int8", "w16", "f16codes", "e4m3"]
MS = [1, 2, 3, 8, 9, 64, 127, 255, 256, 257, 1024, 4096, 4352, 8704]
NS = [16, 200, 256, 768, 3072, 9216, 12288]
KS = [16, 112, 512, 3072, 12288, 131072]


@pytest.fixture(autouse=True)
def restore_options():
    saved = {k: i8.get_option(k) for k in i8.OPTIONS}
    yield
    for k, v in saved.items():
        i8.set_option(k, v)


def _eff(items, slots):
    return items / (math.ceil(items / slots) * slots)


def _check_plan(p, M, N, K, route, m):
    sms = m["sms"]
    pairs = m["pairs"] or sms // 2
    slots = m["skinny_slots"] or 2 * sms
    assert p["num_m"] >= 1 and p["num_n"] >= 1
    # every output row and column in exactly one work item
    if p["kernel"] == "skinny":
        assert p["num_m"] == 1 and p["tile_m"] == M
    else:
        assert (p["num_m"] - 1) * p["tile_m"] < M <= p["num_m"] * p["tile_m"]
    assert (p["num_n"] - 1) * p["tile_n"] < N <= p["num_n"] * p["tile_n"]
    # every K block in exactly one split, no split empty
    assert p["total_kb"] == -(-K // p["block_k"])
    s, kbs = p["splits"], p["kb_per_split"]
    assert s >= 1 and (s - 1) * kbs < p["total_kb"] <= s * kbs
    # the grid fits the machine
    items = p["num_m"] * p["num_n"] * s
    if p["kernel"] == "skinny":
        assert p["grid"] == p["num_n"] * s and p["grid"] <= max(p["num_n"], slots)
    elif p["kernel"] == "tile":
        assert 1 <= p["grid"] <= min(sms, items)
    elif p["kernel"] == "pair_stream_k":
        assert s == 1 and kbs == p["total_kb"] and p["grid"] % 2 == 0
        assert 2 <= p["grid"] <= 2 * pairs
    else:
        assert p["grid"] % 2 == 0 and 2 <= p["grid"] <= 2 * min(pairs, items)
    # the workspace the partials need
    if p["kernel"] == "skinny":
        # the K splits of an N-block form a cluster of at most 8 CTAs and
        # meet in distributed shared memory: no workspace
        assert s <= 8 and p["ws_bytes"] == 0
    elif p["kernel"] == "pair_stream_k":
        tiles = p["num_m"] * p["num_n"]
        arrive = -(-tiles * 16 // 1024) * 1024
        assert p["ws_bytes"] == arrive + p["sk_pairs"] * 256 * 256 * 4   # one slot per sharing pair
        # long K: whole waves on every resident pair first, when there is one
        assert 1 <= p["sk_pairs"] <= p["grid"] // 2
        assert p["sk_waves"] == (tiles // pairs if p["total_kb"] >= 64 else 0)
        if p["sk_waves"] > 0:
            assert p["grid"] == 2 * pairs
    else:
        assert p["ws_bytes"] == (s * M * (-(-N // 4) * 4) * 4 if s > 1 else 0)
    # M blocks fastest when stream-K splits every tile; otherwise N blocks
    # fastest when M > N
    every_tile_split = p["kernel"] == "pair_stream_k" and p["sk_waves"] == 0
    assert p["n_fastest"] == (0 if every_tile_split else 1 if M > N else 0)
    assert (p["model_us"] > 0) == (p["kernel"] == "direct")


def test_every_plan_covers_the_output_once_and_fits_the_machine():
    n = 0
    for m in MACHINES:
        for route in ROUTES:
            for M in MS:
                for N in NS:
                    for K in KS:
                        p = i8.plan_query(M, N, K, route, **m)
                        _check_plan(p, M, N, K, route, m)
                        n += 1
    assert n == len(MACHINES) * len(ROUTES) * len(MS) * len(NS) * len(KS)


def test_kernel_choice_table():
    for M in MS:
        for N in NS:
            for K in KS:
                few = M <= 16
                k8 = i8.plan_query(M, N, K, "int8", **GB300)["kernel"]
                k16 = i8.plan_query(M, N, K, "w16", **GB300)["kernel"]
                if few:
                    assert k8 == k16 == "skinny", (M, N, K)
                    continue
                # CTA pairs for int8 codes once both sides hold a 256 x 256 tile;
                # the pre-widened weights stay on the single-CTA kernel
                assert k8 in (("pair", "pair_stream_k") if M >= 256 and N >= 256 else ("tile",))
                assert k16 == "tile"
                for r in ("f16codes", "e4m3"):
                    assert i8.plan_query(M, N, K, r, **GB300)["kernel"] == "direct"


def test_block_k_per_route():
    assert i8.plan_query(4096, 3072, 3072, "int8", **GB300)["block_k"] == 128
    assert i8.plan_query(4096, 3072, 3072, "e4m3", **GB300)["block_k"] == 128
    assert i8.plan_query(4096, 3072, 3072, "f16codes", **GB300)["block_k"] == 64
    assert i8.plan_query(1, 3072, 3072, "int8", **GB300)["block_k"] == 256


def test_tiled_splits_maximise_the_last_wave():
    """int8 / w16 tiled plans: no split while the tiles fill every worker;
    otherwise the split count maximises the filled fraction of the last wave
    among the counts with at least 4 K blocks per split (smallest on ties)."""
    for route, slots_key in (("int8", "pairs"), ("w16", "sms")):
        for M in (256, 512, 1024, 4096):
            for N in (256, 768, 3072):
                for K in (512, 3072, 12288):
                    i8.set_option("force_splits", 0)
                    p = i8.plan_query(M, N, K, route, **GB300)
                    if p["kernel"] in ("skinny", "pair_stream_k"):
                        continue
                    slots = GB300[slots_key] if p["kernel"] == "pair" else GB300["sms"]
                    tiles = p["num_m"] * p["num_n"]
                    if tiles >= slots:
                        assert p["splits"] == 1
                        continue
                    best = _eff(tiles * p["splits"], slots)
                    for s in range(1, max(1, min(16, p["total_kb"] // 4)) + 1):
                        i8.set_option("force_splits", s)
                        q = i8.plan_query(M, N, K, route, **GB300)
                        assert q["num_m"] * q["num_n"] == tiles
                        e = _eff(tiles * q["splits"], slots)
                        assert e <= best + 1e-9, (route, M, N, K, s)
                        if e > best - 1e-9:
                            assert q["splits"] >= p["splits"]


def test_capped_workspace_plans_fit_the_cap():
    """A workspace cap (the no-alloc entry's fixed 16 MiB array) lowers the
    split count until the partials fit, down to one split that needs none;
    it never rejects a sweep shape.  Without a cap the plan is unchanged, and
    under the cap every plan still covers the output once."""
    cap = 16 << 20
    from w8a8_int8_quantized_i8_gb300 import inputs
    shapes = [(s.M, s.N, s.K) for s in inputs.sweep_shapes()]
    shapes += [(2560, 9216, 3072), (8704, 12288, 3072), (8704, 3072, 12288), (64, 128, 256)]
    lowered = 0
    for m in MACHINES:
        for M, N, K in shapes:
            free = i8.plan_query(M, N, K, "int8", **m)
            p = i8.plan_query(M, N, K, "int8", ws_cap=cap, **m)
            _check_plan(p, M, N, K, "int8", m)
            assert p["ws_bytes"] <= cap, (m, M, N, K, p)
            assert p["splits"] <= free["splits"]
            if free["ws_bytes"] <= cap:
                assert p == free, (m, M, N, K)
            else:
                lowered += 1
                # the largest split count whose partials fit
                if p["kernel"] == "pair" or p["kernel"] == "tile":
                    plane = M * (-(-N // 4) * 4) * 4
                    assert p["splits"] == 1 or p["splits"] * plane <= cap
                    i8.set_option("force_splits", p["splits"] + 1)
                    more = i8.plan_query(M, N, K, "int8", **m)
                    i8.set_option("force_splits", 0)
                    if more["splits"] > p["splits"] and more["splits"] <= free["splits"]:
                        assert more["ws_bytes"] > cap
    assert lowered >= 6        # M = 256 at every (K, N), and M = 1024 at N = 3072


def test_direct_splits_minimise_the_cost_model():
    """Direct plans: no split while the 256 x 256 tiles fill every pair;
    otherwise the chosen split count has the lowest modelled time among the
    counts with at least 4 K blocks per split.  (Up to 16 tokens both routes
    take the weight-streaming kernel instead.)"""
    for route in ("f16codes", "e4m3"):
        for M in (1, 8):
            for N in (768, 3072, 9216):
                p = i8.plan_query(M, N, 3072, route, **GB300)
                assert p["kernel"] == "skinny" and p["ws_bytes"] == 0 and p["block_k"] == 256
        for M in (17, 64, 256, 512, 1024, 4096):
            for N in (768, 3072, 9216):
                for K in (512, 3072, 12288):
                    i8.set_option("force_splits", 0)
                    p = i8.plan_query(M, N, K, route, **GB300)
                    tiles = p["num_m"] * p["num_n"]
                    if tiles >= GB300["pairs"]:
                        assert p["splits"] == 1
                        continue
                    for s in range(1, max(1, min(16, p["total_kb"] // 4)) + 1):
                        i8.set_option("force_splits", s)
                        q = i8.plan_query(M, N, K, route, **GB300)
                        assert q["model_us"] >= p["model_us"] - 1e-9, (route, M, N, K, s)


def test_stream_k_rule():
    # at least half a wave of tiles and a whole-tile wave efficiency below
    # 0.93, at any K: stream-K.  Short K: every tile split, M blocks fastest
    # even where M > N.  Long K: whole waves first, the table's tile order.
    for M, N, K, waves, nf in ((2304, 3072, 3072, 0, 0), (2304, 3072, 12288, 1, 0),
                               (3328, 3072, 12288, 2, 1), (256, 12288, 3072, 0, 0),
                               (1024, 3072, 3072, 0, 0), (8704, 3072, 12288, 5, 1),
                               (1024, 3072, 12288, 0, 0)):
        p = i8.plan_query(M, N, K, "int8", **GB300)
        assert (p["kernel"], p["n_fastest"], p["splits"], p["sk_waves"]) == \
            ("pair_stream_k", nf, 1, waves), (M, N, K)
    p = i8.plan_query(2304, 3072, 12288, "int8", **GB300)
    assert p["grid"] == 2 * GB300["pairs"]
    # high wave efficiency (QKV 2560 x 9216: 360 tiles on 76 pairs, 0.95),
    # fewer than half a wave of tiles (split-K instead), a whole number of
    # waves: no stream-K
    assert i8.plan_query(2560, 9216, 3072, "int8", **GB300)["kernel"] == "pair"
    assert i8.plan_query(74 * 256, 256, 12288, "int8", **GB300)["kernel"] == "pair"
    assert i8.plan_query(2 * GB300["pairs"] * 256, 256, 3072, "int8", **GB300)["kernel"] == "pair"
    for M, N in ((256, 3072), (256, 9216)):
        p = i8.plan_query(M, N, 3072, "int8", **GB300)
        assert p["kernel"] == "pair" and p["splits"] > 1, (M, N)
    # the no-alloc entry's 16 MiB cannot hold the partial slots: falls back
    capped = i8.plan_query(2304, 3072, 12288, "int8", ws_cap=16 << 20, **GB300)
    assert capped["kernel"] == "pair"
    i8.set_option("stream_k", 0)
    assert i8.plan_query(2304, 3072, 12288, "int8", **GB300)["kernel"] == "pair"
    i8.set_option("stream_k", 2)
    assert i8.plan_query(2304, 3072, 3072, "int8", **GB300)["kernel"] == "pair_stream_k"
    assert i8.plan_query(3328, 3072, 12288, "int8", **GB300)["kernel"] == "pair_stream_k"
    i8.set_option("force_splits", 2)      # a forced split count wins over stream-K
    assert i8.plan_query(2304, 3072, 12288, "int8", **GB300)["kernel"] == "pair"


def test_options_change_the_plan():
    i8.set_option("force_splits", 5)
    for route in ROUTES:
        p = i8.plan_query(4096, 3072, 3072, route, **GB300)
        assert p["splits"] == 5, route
    # twelve 256-K stages in 5 splits: 3 stages per split, so 4 splits (none empty)
    one = i8.plan_query(1, 3072, 3072, "int8", **GB300)
    assert (one["splits"], one["kb_per_split"]) == (4, 3)
    assert i8.plan_query(4096, 3072, 16, "int8", **GB300)["splits"] == 1  # one K block
    i8.set_option("force_splits", 0)
    for raster, want in ((1, 0), (2, 1)):
        i8.set_option("raster", raster)
        for M, N in ((8704, 3072), (512, 9216)):
            assert i8.plan_query(M, N, 3072, "int8", **GB300)["n_fastest"] == want
    i8.set_option("raster", 0)
    i8.set_option("skinny_max_m", 0)
    assert i8.plan_query(1, 3072, 3072, "int8", **GB300)["kernel"] == "tile"
    i8.set_option("skinny_max_m", 8)
    assert i8.plan_query(16, 3072, 3072, "int8", **GB300)["kernel"] == "tile"
    i8.set_option("skinny_max_m", 16)
    assert i8.plan_query(16, 3072, 3072, "int8", **GB300)["kernel"] == "skinny"
    i8.set_option("cta_pair", 1)
    assert i8.plan_query(4096, 3072, 3072, "int8", **GB300)["kernel"] == "tile"
    i8.set_option("cta_pair", 2)
    assert i8.plan_query(4096, 9216, 3072, "w16", **GB300)["kernel"] == "pair"
    i8.set_option("cta_pair", 0)
    i8.set_option("tile_n", 128)
    assert i8.plan_query(4096, 3072, 3072, "w16", **GB300)["tile_n"] == 128
    i8.set_option("tile_n", 0)
    i8.set_option("max_ctas", 64)
    assert i8.plan_query(4096, 3072, 3072, "w16", **GB300)["grid"] == 64
    assert i8.plan_query(4096, 3072, 3072, "int8", **GB300)["grid"] == 64


def test_bench_workloads():
    """The plans behind the timed workloads (DiT-XL-like layers at 4096 and
    8704 tokens, GB300 figures)."""
    qkv = i8.plan_query(8704, 9216, 3072, "int8", **GB300)
    assert (qkv["kernel"], qkv["splits"], qkv["n_fastest"], qkv["ws_bytes"]) == ("pair", 1, 0, 0)
    down = i8.plan_query(8704, 3072, 12288, "int8", **GB300)
    assert (down["kernel"], down["splits"], down["n_fastest"], down["sk_waves"]) == ("pair_stream_k", 1, 1, 5)
    one = i8.plan_query(1, 9216, 3072, "int8", **GB300)
    assert (one["kernel"], one["splits"], one["grid"]) == ("skinny", 1, 144)


def test_plan_query_errors():
    lib = i8.load()
    info = i8.PlanInfo()
    call = lambda *a: lib.i8_plan_query(*a)  # noqa: E731
    ok = (64, 64, 64, 0, 152, 0, 0, 0)
    assert call(*ok, ctypes.byref(info)) == 0
    assert call(*ok, None) == 1
    assert call(0, 64, 64, 0, 152, 0, 0, 0, ctypes.byref(info)) == 1
    assert call(64, 0, 64, 0, 152, 0, 0, 0, ctypes.byref(info)) == 1
    assert call(64, 64, 64, 4, 152, 0, 0, 0, ctypes.byref(info)) == 1
    assert call(64, 64, 64, -1, 152, 0, 0, 0, ctypes.byref(info)) == 1
    assert call(64, 64, 64, 0, -1, 0, 0, 0, ctypes.byref(info)) == 1
    assert call(64, 64, 64, 0, 152, -1, 0, 0, ctypes.byref(info)) == 1
    assert call(64, 64, 100, 0, 152, 0, 0, 0, ctypes.byref(info)) == 3
    assert call(64, 64, 131072 + 16, 0, 152, 0, 0, 0, ctypes.byref(info)) == 3
    assert call(1 << 31, 64, 64, 0, 152, 0, 0, 0, ctypes.byref(info)) == 3
    if not torch.cuda.is_available():
        # the current device's figures need a device
        assert call(64, 64, 64, 0, 0, 0, 0, 0, ctypes.byref(info)) == 5
    with pytest.raises(i8.I8Error):
        i8.plan_query(64, 64, 100, "int8", sms=152)
    with pytest.raises(KeyError):
        i8.plan_query(64, 64, 64, "int4", sms=152)


def test_skinny_split_rule():
    """Few tokens: no K split while the N-blocks of 64 weight rows occupy at
    least 90 % of the SMs.  Otherwise the fewest splits that give 5/8 of the
    SMs a CTA, or, when a CTA would then carry more than 12 stages (3072 K),
    the fewest that give every SM a CTA; at most 8, at least 2 stages (512
    K) each, lowered until the grid fits the resident CTA slots (a machine
    described by hand: its clusters assumed to pack those slots fully)."""
    n = 0
    for m in (GB300, dict(sms=152, pairs=74, skinny_slots=152), dict(sms=20, pairs=9, skinny_slots=40)):
        sms, slots = m["sms"], m["skinny_slots"]
        for route in ("int8", "w16", "f16codes", "e4m3"):
            for M in (1, 16):
                for N in (64, 768, 3072, 6144, 8704, 9216, 18432):
                    for K in (256, 1024, 3072, 12288):
                        p = i8.plan_query(M, N, K, route, **m)
                        assert p["kernel"] == "skinny"
                        B, st = -(-N // 64), -(-K // 256)
                        want = 1
                        if 10 * B < 9 * sms:
                            want = -(-max(1, 5 * sms // 8) // B)
                            if -(-st // want) > 12:
                                want = -(-sms // B)
                            want = min(want, max(1, st // 2), 8)
                            while want > 1 and B * want > slots:
                                want -= 1
                        per = -(-st // want)
                        assert (p["splits"], p["kb_per_split"]) == (-(-st // per), per), (m, M, N, K)
                        n += 1
    assert n == 3 * 4 * 2 * 7 * 4
    # the measured cases on GB300 figures (two CTAs per SM); M, N, K
    assert i8.plan_query(1, 3072, 12288, "int8", **GB300)["splits"] == 4
    assert i8.plan_query(1, 9216, 3072, "int8", **GB300)["splits"] == 1
    assert i8.plan_query(16, 3072, 3072, "int8", **GB300)["splits"] == 2
    assert i8.plan_query(1, 768, 3072, "int8", **GB300)["splits"] == 6
    assert i8.plan_query(1, 6144, 2048, "int8", **GB300)["splits"] == 1
