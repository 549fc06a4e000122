"""Pins for the E4M3 (FP8) arm of the CPU oracle, each against something other
than the oracle itself: torch's float8_e4m3fn conversions (an independent
implementation of the OCP E4M3 format), exact rational arithmetic, integer
arithmetic on codes scaled to integers, closed forms and invariants.

A plausible slip in the oracle -- the wrong exponent bias, truncation instead
of ties-to-even, 127 instead of 448, a reciprocal multiply, NaN instead of
saturation, an inexact accumulator, swapped scales -- fails at least one.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from w8a8_int8_quantized_i8_gb300 import inputs


def _torch_decode(codes) -> np.ndarray:
    t = torch.tensor(np.asarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_encode(vals_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(vals_f32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ----------------------------------------------------------------- the format
def test_decode_all_codes_matches_torch(orc):
    want = _torch_decode(np.arange(256))
    got = np.array([orc.e4m3_bits_to_f64(b) for b in range(256)])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(got[~nan], want[~nan])
    assert np.nanmax(got) == 448.0 and np.nanmin(got) == -448.0
    assert got[1] == 2.0 ** -9 and got[8] == 2.0 ** -6


def test_encode_every_bf16_below_saturation_matches_torch(orc):
    # every finite bf16 bit pattern with |v| <= 464 (torch turns larger values
    # into NaN, the oracle saturates; that range is pinned separately)
    pats = np.arange(0, 1 << 16, dtype=np.uint32)
    f = (pats << 16).view(np.float32)
    keep = np.isfinite(f) & (np.abs(f) <= 464.0)
    f = f[keep]
    want = _torch_encode(f)
    got = np.array([orc.f32_to_e4m3_bits(float(v)) for v in f], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {f[bad[:4]]}"


def test_encode_random_fp32_matches_torch(orc):
    rng = np.random.default_rng(7)
    pats = rng.integers(0, 2**32, size=40000, dtype=np.uint64).astype(np.uint32)
    f = pats.view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) <= 464.0)]
    # bias towards the E4M3 range, where rounding decisions happen
    g = (rng.standard_normal(40000) * rng.choice([1e-3, 0.05, 1, 30, 300], 40000)).astype(np.float32)
    g = g[np.abs(g) <= 464.0]
    f = np.concatenate([f, g])
    want = _torch_encode(f)
    got = np.array([orc.f32_to_e4m3_bits(float(v)) for v in f], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_midpoints_round_to_the_even_code(orc):
    vals = _torch_decode(np.arange(0x7F))          # 0 .. 448, increasing
    for c in range(0x7E):
        mid = (vals[c] + vals[c + 1]) / 2          # exact: 5 significant bits
        assert float(np.float32(mid)) == mid
        want = c if c % 2 == 0 else c + 1
        assert orc.f32_to_e4m3_bits(mid) == want, (c, mid)
        assert orc.f32_to_e4m3_bits(-mid) == 0x80 | want
        # a hair either side of the midpoint decides by distance
        lo = float(np.nextafter(np.float32(mid), np.float32(0)))
        hi = float(np.nextafter(np.float32(mid), np.float32(1e9)))
        assert orc.f32_to_e4m3_bits(lo) == c
        assert orc.f32_to_e4m3_bits(hi) == c + 1


def test_saturation_and_specials(orc):
    for v in (448.0, 449.0, 463.99, 464.0, 464.01, 480.0, 1e4, 3.4e38, math.inf):
        assert orc.f32_to_e4m3_bits(v) == 0x7E, v
        assert orc.f32_to_e4m3_bits(-v) == 0xFE, v
    assert orc.f32_to_e4m3_bits(math.nan) == 0x7F
    assert orc.f32_to_e4m3_bits(0.0) == 0x00
    assert orc.f32_to_e4m3_bits(-0.0) == 0x80
    # underflow: half the smallest subnormal is a tie with 0 (even), above it 2^-9
    assert orc.f32_to_e4m3_bits(2.0 ** -10) == 0x00
    assert orc.f32_to_e4m3_bits(float(np.nextafter(np.float32(2.0 ** -10), np.float32(1)))) == 0x01
    assert orc.f32_to_e4m3_bits(1e-30) == 0x00
    assert orc.f32_to_e4m3_bits(-1e-30) == 0x80


# ----------------------------------------------------------------- quantizer
def _row_bits(vals):
    return inputs.bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


def test_quant_rows_e4m3_exact_rational(orc):
    g = torch.Generator().manual_seed(11)
    x = torch.randn(24, 300, generator=g)
    x[:, 7] *= 20.0
    x[3] *= 1e-30                                   # tiny row (subnormal scale)
    x[5] = 0.0
    x[6, :] = 0.0
    x[6, 4] = -0.0                                  # zero row with a negative zero
    bits = inputs.bits(x.to(torch.bfloat16))
    q, s = orc.quant_rows_e4m3(bits)
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    for r in range(x.shape[0]):
        amax = float(np.abs(xf[r]).max())
        if amax == 0.0:
            assert s[r] == 0.0 and (q[r] == 0).all()
            continue
        sr = float(s[r])
        # the fp32 scale is the float nearest to amax / 448
        exact = Fraction(amax) / 448
        cand = [np.float32(sr), np.nextafter(np.float32(sr), np.float32(0)),
                np.nextafter(np.float32(sr), np.float32(1))]
        assert min(abs(Fraction(float(c)) - exact) for c in cand) == abs(Fraction(sr) - exact)
        # every code is the E4M3 value nearest to the fp32 quotient x / s
        t = (xf[r] / np.float32(sr)).astype(np.float32)   # IEEE fp32 division
        assert np.array_equal(q[r], _torch_encode(np.clip(t, -464, 464)))
        # the absmax element lands on +-448
        dec = _torch_decode(q[r])
        assert np.abs(dec).max() == 448.0


def test_quant_rows_e4m3_sign_symmetry_and_monotone(orc):
    g = torch.Generator().manual_seed(12)
    x = torch.randn(4, 512, generator=g)
    b = inputs.bits(x.to(torch.bfloat16))
    q, s = orc.quant_rows_e4m3(b)
    qn, sn = orc.quant_rows_e4m3(b ^ np.uint16(0x8000))
    assert np.array_equal(s, sn)
    assert np.array_equal(qn, q ^ np.uint8(0x80))
    xf = (b.astype(np.uint32) << 16).view(np.float32)
    for r in range(4):
        o = np.argsort(xf[r], kind="stable")
        d = _torch_decode(q[r][o])
        assert (np.diff(d) >= 0).all()


def test_quant_rows_e4m3_scale_closed_form(orc):
    # amax = 448 gives s = 1 exactly, so codes are E4M3(x) itself
    vals = [448.0, -3.0, 0.1, 17.0, -0.0078125, 300.0]
    q, s = orc.quant_rows_e4m3(_row_bits([vals]))
    assert s[0] == 1.0
    xf = (_row_bits(vals).astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(q[0], _torch_encode(xf))


# ----------------------------------------------------------------- GEMM
def _codes_as_int(c: np.ndarray) -> np.ndarray:
    """E4M3 codes as exact integers in units of 2^-9 (via torch's decode)."""
    v = _torch_decode(c) * 512.0
    assert (v == np.round(v)).all()
    return v.astype(np.int64)


def test_gemm_e4m3_exact_against_integer_arithmetic(orc):
    rng = np.random.default_rng(5)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    for (M, N, K) in [(3, 5, 7), (16, 9, 256), (2, 3, 4096)]:
        a = rng.choice(codes, size=(M, K))
        w = rng.choice(codes, size=(N, K))
        want = _codes_as_int(a) @ _codes_as_int(w).T          # units of 2^-18, exact
        got = orc.gemm_e4m3_f64(a, w)
        assert np.array_equal(got * 2.0 ** 18, want.astype(np.float64))
        assert (np.abs(want) < 2 ** 53).all()
        got_abs = orc.gemm_e4m3_f64(a, w, absval=True)
        want_abs = np.abs(_codes_as_int(a)) @ np.abs(_codes_as_int(w)).T
        assert np.array_equal(got_abs * 2.0 ** 18, want_abs.astype(np.float64))


def test_gemm_e4m3_closed_forms(orc):
    K = 131072
    ones = np.full((1, K), 0x38, dtype=np.uint8)            # 1.0
    assert orc.gemm_e4m3_f64(ones, ones)[0, 0] == K
    big = np.full((1, K), 0x7E, dtype=np.uint8)             # 448
    assert orc.gemm_e4m3_f64(big, big)[0, 0] == 448.0 * 448.0 * K
    neg = big | np.uint8(0x80)
    assert orc.gemm_e4m3_f64(big, neg)[0, 0] == -448.0 * 448.0 * K
    tiny = np.full((1, K), 0x01, dtype=np.uint8)            # 2^-9
    assert orc.gemm_e4m3_f64(tiny, tiny)[0, 0] == K * 2.0 ** -18
    # identity weights (N = K) reproduce the decoded rows: catches a transpose
    rng = np.random.default_rng(9)
    a = rng.integers(0, 0x7E, size=(4, 32)).astype(np.uint8)
    eye = np.where(np.eye(32, dtype=bool), 0x38, 0x00).astype(np.uint8)
    assert np.array_equal(orc.gemm_e4m3_f64(a, eye), _torch_decode(a))
    with pytest.raises(ValueError):
        orc.gemm_e4m3_f64(np.zeros((1, 131088), np.uint8), np.zeros((1, 131088), np.uint8))


# ----------------------------------------------------------------- epilogue
def test_dequant_f64acc_matches_int32_epilogue_on_integers(orc):
    rng = np.random.default_rng(3)
    acc = rng.integers(-(2 ** 30), 2 ** 30, size=(6, 40)).astype(np.int32)
    sa = rng.random(6).astype(np.float32) * 1e-3
    sw = rng.random(40).astype(np.float32) * 1e-2
    bias = inputs.bits(torch.randn(40, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16))
    want = orc.dequant_bias(acc, sa, sw, bias)
    got = orc.dequant_bias_f64acc(acc.astype(np.float64), sa, sw, bias)
    assert np.array_equal(got, want)
    # and within one bf16 ulp of an fp64 evaluation
    bf = (bias.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = acc.astype(np.float64) * sa[:, None] * sw[None, :] + bf[None, :]
    y = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert (np.abs(y - ref) <= 2.0 ** -8 * np.abs(ref) * 1.01 + 1e-30).all()


def test_linear_e4m3_tracks_the_unquantized_product(orc):
    g = torch.Generator().manual_seed(21)
    x = torch.randn(32, 256, generator=g)
    w = torch.randn(48, 256, generator=g) * 0.02
    b = torch.randn(48, generator=g) * 0.01
    xb, wb, bb = (inputs.bits(t.to(torch.bfloat16)) for t in (x, w, b))
    r = orc.linear_e4m3(xb, wb, bb)
    xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wf = (wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bf = (bb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = xf @ wf.T + bf
    y = (r["y"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    cos = (y * ref).sum() / np.linalg.norm(y) / np.linalg.norm(ref)
    # E4M3 keeps 4 significant bits: per-element relative error ~2^-5, so the
    # layer output stays within a few per cent and the cosine near 1
    assert cos > 0.998
    assert np.abs(y - ref).max() < 0.1 * np.abs(ref).max()
