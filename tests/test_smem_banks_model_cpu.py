"""Shared-memory bank use of the on-chip widening, modelled on the CPU.

The int8-code GEMM kernels widen each staged int8 block to fp16 in shared
memory: converter thread item i reads 16 codes (one 16-byte chunk of a
128-byte swizzled int8 row) and writes 32 bytes (two chunks of a 128-byte
swizzled fp16 row).  With the 128-byte swizzle, logical chunk c of row r sits
at physical chunk c ^ (r & 7).  A 128-bit shared access of a warp is served
in four phases of eight lanes; a phase takes one wavefront when its eight
16-byte chunks fall in eight different 4-bank groups.  This model computes
the converters' addresses as the kernels do (item -> row, chunk; one item per
lane; lanes of a warp on consecutive items) for every configuration the
library builds, and counts the wavefronts of each access: every one is
conflict-free, 4 wavefronts per warp access, the minimum.  So the extra
wavefronts that profiling attributes to these accesses do not come from the
addresses themselves.
"""
import os

import pytest

BK8, BK16 = 128, 64
CONV_THREADS = 6 * 32


def conv_item(i, bm, bn, conv_a, conv_b):
    a_items = bm * 4 if conv_a else 0
    a8 = bm * BK8 if conv_a else 0
    a16 = bm * BK16 * 2
    if i < a_items:
        region8, region16, rows, idx = 0, 0, bm, i
    else:
        region8, region16, rows, idx = a8, a16, bn, i - a_items
    cl, r = idx // rows, idx % rows
    x = r & 7
    return region8 + r * 128 + ((cl ^ x) << 4), region16 + r * 128 + (((2 * cl) ^ x) << 4)


def wavefronts(addrs):
    """Wavefronts of one warp's 128-bit shared access (None = inactive lane)."""
    total = 0
    for ph in range(4):
        banks = {}
        for a in addrs[8 * ph:8 * ph + 8]:
            if a is None:
                continue
            assert a % 16 == 0
            for w in range(4):
                word = a // 4 + w
                banks.setdefault(word % 32, set()).add(word)
        total += max((len(v) for v in banks.values()), default=0)
    return total


CONFIGS = [
    # (name, BM rows of A staged, BN rows of B staged, A widened, B widened)
    ("pair kernel, int8 weights", 128, 128, True, True),
    ("pair kernel, pre-widened weights", 128, 128, True, False),
    ("1-CTA kernel, 128-wide tile, int8 weights", 128, 128, True, True),
    ("1-CTA kernel, 256-wide tile, int8 weights", 128, 256, True, True),
    ("1-CTA kernel, pre-widened weights", 128, 256, True, False),
]


@pytest.mark.parametrize("name,bm,bn,conv_a,conv_b", CONFIGS)
def test_widening_accesses_are_conflict_free(name, bm, bn, conv_a, conv_b):
    items = (bm * 4 if conv_a else 0) + (bn * 4 if conv_b else 0)
    ipt = -(-items // CONV_THREADS)
    checked = 0
    for warp in range(CONV_THREADS // 32):
        for j in range(ipt):
            lanes = [warp * 32 + lane + j * CONV_THREADS for lane in range(32)]
            its = [conv_item(i, bm, bn, conv_a, conv_b) if i < items else None for i in lanes]
            if all(t is None for t in its):
                continue
            for h in range(2):                          # the two 64-K halves of the block
                loads = [None if t is None else t[0] ^ (h << 6) for t in its]
                stores0 = [None if t is None else t[1] for t in its]
                stores1 = [None if t is None else t[1] ^ 16 for t in its]
                for acc in (loads, stores0, stores1):
                    active_phases = sum(any(a is not None for a in acc[8 * p:8 * p + 8])
                                        for p in range(4))
                    assert wavefronts(acc) == active_phases, (name, warp, j, h)
                    checked += 1
    assert checked > 0


def test_every_code_is_widened_once_to_its_place():
    """The items cover every 16-code chunk of the int8 stage once (both
    64-K halves), and each lands in the two fp16 chunks of the same row that
    hold the same K positions of its half's sub-tile."""
    for name, bm, bn, conv_a, conv_b in CONFIGS:
        a8 = bm * BK8 if conv_a else 0
        a16 = bm * BK16 * 2
        items = (bm * 4 if conv_a else 0) + (bn * 4 if conv_b else 0)
        seen = set()
        for i in range(items):
            src, dst = conv_item(i, bm, bn, conv_a, conv_b)
            in_a = i < (bm * 4 if conv_a else 0)
            s_rel = src - (0 if in_a else a8)
            d_rel = dst - (0 if in_a else a16)
            r8, d_row = s_rel // 128, d_rel // 128
            assert r8 == d_row
            x = r8 & 7
            for h in range(2):
                k8 = 16 * ((((s_rel % 128) >> 4) ^ (4 * h)) ^ x)          # first K of the int8 chunk
                k16 = [8 * ((((d_rel ^ e) % 128) >> 4) ^ x) for e in (0, 16)]  # first K of each fp16 chunk
                assert k16 == [k8 - 64 * h, k8 - 64 * h + 8], (name, i, h)
                key = (in_a, r8, k8)
                assert key not in seen
                seen.add(key)
        assert len(seen) == 2 * items                 # 8 chunks of 16 codes per 128-byte row


def test_model_restates_the_kernel_source():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "w8a8_int8_quantized_i8_gb300", "csrc", "gemm.cuh")
    with open(path) as fh:
        src = " ".join(fh.read().split())
    for text in ["const int cl = idx / rows; const int r = idx % rows; const int x = r & 7;",
                 "it.src = static_cast<uint32_t>(region8 + r * 128 + ((cl ^ x) << 4));",
                 "it.dst = static_cast<uint32_t>(region16 + r * 128 + (((2 * cl) ^ x) << 4));"]:
        assert text in src, text
