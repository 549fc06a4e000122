"""Pins for the oracle's producer steps (LayerNorm without affine, GELU in erf
form, and the single fp64 -> bf16 rounding they share), each against
something other than the oracle: torch's fp64 layer_norm / gelu, closed forms,
invariants and the ordering of neighbouring bf16 values.

A plausible slip -- a biased variance (K - 1), eps outside the square root, a
double rounding through fp32, the tanh form of GELU, the cancelling
1 + erf(x / sqrt 2) in the negative tail, a truncating round -- fails at least
one of them.
"""
import math

import numpy as np
import pytest
import torch

scipy = pytest.importorskip("scipy")
import scipy.special  # noqa: E402

from w8a8_int8_quantized_i8_gb300 import inputs


def _f64(bits: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):          # NaN patterns stay NaN
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------- rounding
def test_f64_to_bf16_is_the_nearest_neighbour(orc):
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                           [1.0, -1.0, 3.0e38, 1e-40, -2.5e-39]])
    for v in vals:
        b = orc.f64_to_bf16_bits(float(v))
        y = float(_f64(np.array([b], np.uint16))[0])
        # the two bf16 neighbours of the result, by bit adjacency
        up = float(_f64(np.array([b + 1], np.uint16))[0]) if (b & 0x7FFF) < 0x7F7F else math.inf
        dn = float(_f64(np.array([b - 1], np.uint16))[0]) if (b & 0x7FFF) > 0 else 0.0
        assert abs(y - v) <= abs(up - v) and abs(y - v) <= abs(dn - v), v
        assert math.copysign(1.0, y) == math.copysign(1.0, v) or y == 0.0


def test_f64_to_bf16_ties_to_even_and_single_rounding(orc):
    # exact midpoints between neighbouring bf16 values go to the even pattern
    for b in (0x3F80, 0x3F81, 0x4000, 0x0001, 0x7F00, 0xBF83):
        lo = float(_f64(np.array([b], np.uint16))[0])
        hi = float(_f64(np.array([b + 1], np.uint16))[0])
        mid = (lo + hi) / 2
        assert orc.f64_to_bf16_bits(mid) == (b if b % 2 == 0 else b + 1)
        # a midpoint plus less than an fp32 ulp: a double rounding through
        # fp32 would land on the midpoint and go to even; one rounding goes up
        above = mid + math.copysign(abs(mid) * 2.0 ** -30, mid)   # away from zero
        assert orc.f64_to_bf16_bits(above) == b + 1, hex(b)
    # values exactly representable in fp32 agree with torch's fp32 -> bf16 cast
    f = np.random.default_rng(3).standard_normal(5000).astype(np.float32)
    want = inputs.bits(torch.from_numpy(f).to(torch.bfloat16))
    got = np.array([orc.f64_to_bf16_bits(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, want)


# ----------------------------------------------------------------- LayerNorm
def _torch_ln(bits: np.ndarray, eps: float) -> np.ndarray:
    x = torch.from_numpy(_f64(bits))
    return torch.nn.functional.layer_norm(x, (x.shape[-1],), eps=eps).numpy()


def test_layernorm_matches_torch_fp64(orc):
    g = torch.Generator().manual_seed(4)
    x = inputs.activations(40, 3072, g)
    x[3] = (x[3].float() * 1e-3 + 7.0).to(torch.bfloat16)      # large mean, small spread
    bits = inputs.bits(x)
    y = orc.layernorm_rows(bits, 1e-6)
    ref = _torch_ln(bits, 1e-6)
    got = _f64(y)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) * (1 + 1e-9) + 1e-30)
    # torch's value rounded once is the oracle's value except at near-midpoints
    exact = np.array([[orc.f64_to_bf16_bits(v) for v in row] for row in ref[:4]], dtype=np.uint16)
    assert (exact == y[:4]).mean() > 0.999


def test_layernorm_closed_forms(orc):
    K = 256
    alt = np.where(np.arange(K) % 2 == 0, 1.0, -1.0).astype(np.float32)
    rows = np.stack([alt, alt * 3.0, np.full(K, 2.5, np.float32), np.zeros(K, np.float32)])
    bits = inputs.bits(torch.from_numpy(rows).to(torch.bfloat16))
    y = _f64(orc.layernorm_rows(bits, 1e-6))
    # mean 0, variance a^2: y = +-a / sqrt(a^2 + eps), which is +-1 in bf16
    assert np.array_equal(y[0], alt.astype(np.float64))
    assert np.array_equal(y[1], alt.astype(np.float64))
    # constant and zero rows: x - mu = 0
    assert (y[2] == 0).all() and (y[3] == 0).all()
    # eps inside the square root: a row with variance 1e-6 and eps 1e-6 maps
    # to +-1 / sqrt(2)
    small = np.where(np.arange(K) % 2 == 0, 1e-3, -1e-3)
    sb = np.array([[orc.f64_to_bf16_bits(v) for v in small]], dtype=np.uint16)
    xs = _f64(sb)[0]
    var = float(np.mean((xs - xs.mean()) ** 2))
    want = (xs - xs.mean()) / math.sqrt(var + 1e-6)
    got = _f64(orc.layernorm_rows(sb, 1e-6))[0]
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want))
    assert abs(abs(got[0]) - 1 / math.sqrt(1 + 1e-6 / var)) < 0.01


def test_layernorm_invariants(orc):
    g = torch.Generator().manual_seed(6)
    x = inputs.activations(16, 1024, g, "gelu")
    bits = inputs.bits(x)
    y = _f64(orc.layernorm_rows(bits, 0.0))
    assert np.all(np.abs(y.mean(axis=1)) < 1e-3)
    assert np.all(np.abs(y.var(axis=1) - 1.0) < 1e-2)         # biased variance (1/K)
    # scaling the row by 2 (exact in bf16) leaves the output unchanged when eps = 0
    y2 = _f64(orc.layernorm_rows(inputs.bits((x.float() * 2).to(torch.bfloat16)), 0.0))
    assert np.array_equal(y, y2)


# ----------------------------------------------------------------- GELU
def test_gelu_matches_torch_fp64_and_identity(orc):
    vals = np.unique(np.concatenate([
        np.arange(0, 1 << 16, 7, dtype=np.uint32)]).astype(np.uint16))
    xf = _f64(vals)
    keep = np.isfinite(xf) & (np.abs(xf) < 1e4)
    vals = vals[keep]
    y = orc.gelu_rows(vals[None, :])[0]
    xv = _f64(vals)
    # torch's fp64 gelu evaluates 1 + erf(x / sqrt 2), which loses relative
    # accuracy as x falls (about 1e-16 / Phi(x)) and cancels to 0 below about
    # x = -8.3; below x = -5 the pin is x * Phi(x) from scipy's normal CDF
    ref = torch.nn.functional.gelu(torch.from_numpy(xv), approximate="none").numpy()
    tail = xv < -5.0
    ref[tail] = xv[tail] * scipy.special.ndtr(xv[tail])
    got = _f64(y)
    tol = 2.0 ** -8 * np.abs(ref) * (1 + 1e-9) + 2.0 ** -134   # half the subnormal spacing
    assert np.all(np.abs(got - ref) <= tol)
    # the tail is not flushed: gelu(-9.25) = -1.0e-19, gelu(-13.25) ~ -2.6e-39
    t = inputs.bits(torch.tensor([[-9.25, -13.25]]).to(torch.bfloat16))
    yt = _f64(orc.gelu_rows(t))[0]
    assert -1.1e-19 < yt[0] < -0.9e-19 and yt[1] < 0
    # the tanh form differs by far more than that on [1, 3]
    x = np.linspace(1, 3, 64)
    tanh_form = 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))
    erf_form = 0.5 * x * (1 + np.array([math.erf(v / math.sqrt(2)) for v in x]))
    assert np.abs(tanh_form - erf_form).max() > 1e-4
    # gelu(x) - gelu(-x) = x, up to the two roundings
    pos = vals[(xf[keep] > 0) & (xf[keep] < 100)]
    yp = _f64(orc.gelu_rows(pos[None, :])[0])
    yn = _f64(orc.gelu_rows((pos | np.uint16(0x8000))[None, :])[0])
    xp = _f64(pos)
    assert np.all(np.abs(yp - yn - xp) <= 2.0 ** -8 * (np.abs(yp) + np.abs(yn)) + 2.0 ** -133)
    assert orc.gelu_rows(np.array([[0x0000, 0x8000]], np.uint16)).tolist() == [[0x0000, 0x8000]]
    big = inputs.bits(torch.tensor([[8.0, 100.0, 1000.0]]).to(torch.bfloat16))
    assert np.array_equal(orc.gelu_rows(big), big)


def test_producer_quant_composes(orc):
    g = torch.Generator().manual_seed(8)
    x = inputs.activations(8, 512, g)
    bits = inputs.bits(x)
    y, q, s = orc.producer_quant_rows(bits, "layernorm", "int8")
    q2, s2 = orc.quant_rows(orc.layernorm_rows(bits))
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    y, q, s = orc.producer_quant_rows(bits, "gelu", "e4m3")
    q3, s3 = orc.quant_rows_e4m3(orc.gelu_rows(bits))
    assert np.array_equal(q, q3) and np.array_equal(s, s3)
