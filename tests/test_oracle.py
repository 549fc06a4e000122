"""Pins for the CPU oracle, each against something other than the oracle itself.

The pages print no tensors, scales or outputs for a worked example, so the
pins are: exact rational arithmetic (``fractions.Fraction``), closed forms
derived by hand (``tests/golden/``), library routines (numpy int64 matmul,
torch's fp32->bf16 cast), brute force on tiny inputs, and invariants.  They
are chosen so that a plausible slip in the oracle -- 128 instead of 127, a
truncating round, a reciprocal multiply, a transposed operand, swapped scales,
a dropped bias -- fails at least one of them.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from w8a8_int8_quantized_i8_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def _bf16_bits(vals):
    return inputs.bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


def _ulp32(x: float) -> Fraction:
    """Spacing of float32 numbers at |x| (x a nonzero float32)."""
    _, e = math.frexp(abs(x))            # |x| = m * 2**e, m in [0.5, 1)
    e = max(e, -125)                     # subnormal range has a fixed spacing
    return Fraction(2) ** (e - 24)


# ----------------------------------------------------------------- bf16 rounding
def test_f32_to_bf16_matches_torch_cast(orc):
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    pats = pats[(pats & 0x7F800000) != 0x7F800000]
    edge = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x00008000, 0x00018000,
                     0x7F7FFFFF, 0xFF7FFFFF, 0x7F7F8000, 0x00000001, 0x80000000,
                     0x00000000, 0x3F800001, 0x3F807FFF], dtype=np.uint32)
    pats = np.concatenate([pats, edge])
    f = pats.view(np.float32)
    want = inputs.bits(torch.from_numpy(f.copy()).to(torch.bfloat16))
    got = np.array([orc.f32_to_bf16_bits(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_widening_is_exact(orc):
    for b in (0x0000, 0x8000, 0x3F80, 0xC2FE, 0x0001, 0x7F7F, 0x4B00):
        want = struct.unpack("<f", struct.pack("<I", b << 16))[0]
        assert orc.bf16_bits_to_f32(b) == want


# ----------------------------------------------------------------- quantizer
def test_quant_golden_ties(orc):
    with open(os.path.join(GOLDEN, "quant_ties.json")) as fh:
        gold = json.load(fh)
    for row in gold["rows"]:
        q, s = orc.quant_rows(_bf16_bits(row["x"])[None, :])
        assert float(s[0]) == row["scale"]
        assert q[0].tolist() == row["q"]


def test_quant_multiples_of_power_of_two_scale(orc):
    # absmax = 127 * 2^e makes the scale exactly 2^e; x = j * 2^e must give j.
    for e in (-6, -1, 0, 3):
        step = 2.0 ** e
        xs = [j * step for j in range(-127, 128)]
        q, s = orc.quant_rows(_bf16_bits(xs)[None, :])
        assert float(s[0]) == step
        assert q[0].tolist() == list(range(-127, 128))


def test_quant_zero_row(orc):
    q, s = orc.quant_rows(np.zeros((3, 48), dtype=np.uint16))
    assert np.all(q == 0) and np.all(s == 0)
    q, s = orc.quant_rows(np.full((1, 16), 0x8000, dtype=np.uint16))  # -0.0
    assert np.all(q == 0) and s[0] == 0


def _check_row_exact(xbits_row, q_row, s):
    """Exact-rational pins for the scale and every code of one row."""
    xs = [struct.unpack("<f", struct.pack("<I", int(b) << 16))[0] for b in xbits_row]
    amax = max(abs(v) for v in xs)
    if amax == 0:
        assert s == 0 and all(int(c) == 0 for c in q_row)
        return
    s = float(s)
    assert s == _f32(s)
    # (1) the scale is the float32 nearest to amax/127 (half-ulp bound)
    assert abs(Fraction(s) - Fraction(amax) / 127) <= _ulp32(s) / 2
    # (2) every code lies within 1/2 (+ the quotient's own rounding) of
    #     x / scale, inside +-127, and the absmax element maps to +-127
    tol = Fraction(1, 2) + Fraction(1, 2**16)
    for v, c in zip(xs, q_row):
        c = int(c)
        assert -127 <= c <= 127
        assert abs(Fraction(v) / Fraction(s) - c) <= tol, (v, s, c)
        if abs(v) == amax:
            assert c == (127 if v > 0 else -127)


def test_quant_exact_rational_random_rows(orc):
    x = inputs.activations(24, 320, torch.Generator().manual_seed(7), outliers=True)
    xb = inputs.bits(x)
    q, s = orc.quant_rows(xb)
    for r in range(xb.shape[0]):
        _check_row_exact(xb[r], q[r], s[r])


def test_quant_exhaustive_bf16_with_unit_absmax(orc):
    # Every finite bf16 value in [-1, 1] in one row whose absmax is 1.
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = (allb.astype(np.uint32) << 16).view(np.float32)
    keep = np.isfinite(f) & (np.abs(f) <= 1.0)
    row = allb[keep]
    q, s = orc.quant_rows(row[None, :])
    _check_row_exact(row, q[0], s[0])
    # a row with a subnormal absmax: no flush to zero anywhere
    sub = np.array([0x0001, 0x8003, 0x0005, 0x007F, 0x8040], dtype=np.uint16)
    q2, s2 = orc.quant_rows(sub[None, :])
    assert s2[0] > 0
    _check_row_exact(sub, q2[0], s2[0])


def test_quant_uses_true_division(orc):
    # Find (x, absmax) where rounding x * (1/scale) disagrees with rounding the
    # correctly rounded quotient; the oracle must follow the division.
    rng = np.random.default_rng(3)
    found = 0
    for _ in range(200000):
        amax = inputs.bits(torch.tensor([float(rng.uniform(0.5, 4.0))]).to(torch.bfloat16))[0]
        amax_f = np.float32(struct.unpack("<f", struct.pack("<I", int(amax) << 16))[0])
        s = np.float32(amax_f / np.float32(127.0))
        j = rng.integers(-126, 126)
        xb = inputs.bits(torch.tensor([float((j + 0.5) * s)]).to(torch.bfloat16))[0]
        xf = np.float32(struct.unpack("<f", struct.pack("<I", int(xb) << 16))[0])
        if abs(xf) > amax_f:
            continue
        by_div = np.rint(np.float32(xf / s))
        by_rcp = np.rint(np.float32(xf * np.float32(np.float32(1.0) / s)))
        if by_div != by_rcp:
            q, sc = orc.quant_rows(np.array([[amax, xb]], dtype=np.uint16))
            assert float(sc[0]) == float(s)
            assert int(q[0, 1]) == int(by_div)
            found += 1
            if found >= 5:
                break
    assert found >= 1, "no division/reciprocal disagreement found to pin"


def test_quant_scale_is_absmax_over_127_not_128(orc):
    q, s = orc.quant_rows(_bf16_bits([1.0, -0.5, 0.25])[None, :])
    assert float(s[0]) == _f32(1.0 / 127.0)
    assert q[0].tolist() == [127, -64, 32]   # -63.5 -> -64 (even), 31.75 -> 32


# ----------------------------------------------------------------- GEMM
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 5, 33), (16, 24, 48), (33, 17, 256)])
def test_gemm_matches_numpy_int64(orc, M, N, K):
    a = inputs.random_int8(M, K, seed=M * 1000 + K).numpy()
    w = inputs.random_int8(N, K, seed=N * 1000 + K + 1).numpy()
    got = orc.gemm_s32(a, w)
    want = a.astype(np.int64) @ w.astype(np.int64).T
    assert got.dtype == np.int32
    assert np.array_equal(got.astype(np.int64), want)


def test_gemm_golden_closed_forms(orc):
    with open(os.path.join(GOLDEN, "gemm_closed_forms.json")) as fh:
        gold = json.load(fh)
    for case in gold["cases"]:
        K = case["K"]
        a = np.full((2, K), case["a_value"], dtype=np.int8)
        w = np.full((3, K), case["w_value"], dtype=np.int8)
        c = orc.gemm_s32(a, w)
        assert np.all(c == case["acc"]), case["name"]


def test_gemm_identity_weights_reproduce_rows(orc):
    K = 64
    a = inputs.random_int8(9, K, seed=11).numpy()
    eye = np.eye(K, dtype=np.int8)
    assert np.array_equal(orc.gemm_s32(a, eye), a.astype(np.int32))
    # a permutation matrix picks columns: catches a transposed operand
    perm = np.random.default_rng(0).permutation(K)
    assert np.array_equal(orc.gemm_s32(a, eye[perm]), a[:, perm].astype(np.int32))


def test_gemm_rejects_overflowing_k(orc):
    a = np.ones((1, 131073), dtype=np.int8)
    with pytest.raises(ValueError):
        orc.gemm_s32(a, a)


# ----------------------------------------------------------------- epilogue
def test_epilogue_within_one_bf16_ulp_of_fp64(orc):
    rng = np.random.default_rng(5)
    M, N = 37, 29
    acc = rng.integers(-2**30, 2**30, size=(M, N), dtype=np.int64).astype(np.int32)
    acc[0, :] = 0
    s_a = rng.uniform(1e-4, 0.2, size=M).astype(np.float32)
    s_w = rng.uniform(1e-6, 1e-3, size=N).astype(np.float32)
    bias = inputs.bits(torch.from_numpy(rng.normal(0, 0.5, size=N).astype(np.float32)).to(torch.bfloat16))
    y = orc.dequant_bias(acc, s_a, s_w, bias)
    yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bf = (bias.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = (acc.astype(np.float64) * s_a[:, None].astype(np.float64)
           * s_w[None, :].astype(np.float64) + bf[None, :])
    assert np.all(np.abs(yf - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)


def test_epilogue_zero_accumulator_gives_bias(orc):
    N = 40
    bias = _bf16_bits(np.linspace(-3, 3, N).tolist())
    y = orc.dequant_bias(np.zeros((3, N), np.int32), np.array([0.5, 0.0, 3.0], np.float32),
                         np.full(N, 0.01, np.float32), bias)
    assert np.array_equal(y, np.broadcast_to(bias, (3, N)))


def test_epilogue_unit_scales_is_acc_plus_bias(orc):
    rng = np.random.default_rng(9)
    M, N = 8, 64
    acc = rng.integers(-300, 300, size=(M, N)).astype(np.int32)
    bias_f = torch.from_numpy(rng.normal(0, 2, size=N).astype(np.float32)).to(torch.bfloat16)
    want = inputs.bits((torch.from_numpy(acc).to(torch.float32)
                        + bias_f.to(torch.float32)[None, :]).to(torch.bfloat16))
    y = orc.dequant_bias(acc, np.ones(M, np.float32), np.ones(N, np.float32), inputs.bits(bias_f))
    assert np.array_equal(y, want)


def test_epilogue_scale_roles_are_row_and_column(orc):
    # per-token scale varies along rows, per-channel along columns
    acc = np.ones((2, 3), np.int32) * 64
    y = orc.dequant_bias(acc, np.array([1.0, 2.0], np.float32),
                         np.array([1.0, 0.5, 0.25], np.float32), None)
    yf = (y.astype(np.uint32) << 16).view(np.float32)
    assert yf.tolist() == [[64.0, 32.0, 16.0], [128.0, 64.0, 32.0]]


def test_epilogue_no_bias_matches_torch_fp32_steps(orc):
    rng = np.random.default_rng(10)
    M, N = 16, 24
    acc = rng.integers(-2**28, 2**28, size=(M, N)).astype(np.int32)
    s_a = rng.uniform(1e-3, 1.0, size=M).astype(np.float32)
    s_w = rng.uniform(1e-5, 1e-2, size=N).astype(np.float32)
    t = torch.from_numpy(acc).to(torch.float32) * torch.from_numpy(s_a)[:, None]
    t = t * torch.from_numpy(s_w)[None, :]
    assert np.array_equal(orc.dequant_bias(acc, s_a, s_w, None), inputs.bits(t.to(torch.bfloat16)))


# ----------------------------------------------------------------- whole path
def test_linear_tiny_config_close_to_unquantized(orc):
    d = inputs.linear_inputs(inputs.TINY)
    out = orc.linear(inputs.bits(d["x"]), inputs.bits(d["w"]), inputs.bits(d["bias"]))
    y = (out["y"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = (d["x"].double() @ d["w"].double().T + d["bias"].double()).numpy()
    cos = float((y * ref).sum() / (np.linalg.norm(y) * np.linalg.norm(ref)))
    assert cos > 0.999
    assert np.isfinite(y).all()
    xf = d["x"].float().numpy()
    assert np.all(np.abs(out["aq"] * out["s_a"][:, None] - xf) <= out["s_a"][:, None] * 0.5001)
