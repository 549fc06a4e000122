"""The E4M3 arm's accumulator tolerance, modelled on the CPU.

The E4M3 GEMM (the FP8 arm the pages set against INT8: "Realizing Native INT8
Compute for Diffusion Transformers on Consumer GPUs", abstract) accumulates in
fp32 on the tensor cores, 32 products per MMA step, and the tests allow
  |acc - S| <= (ceil(K / 32) + 1) * 2 * 2^-24 * P,   P = sum_k |a_k w_k|,
S the exact sum.  The derivation: every E4M3 product is exact (at most 8
significant bits) and a block of 32 is exact in fp32 range, so each step adds
one rounding of a partial sum of magnitude <= P; two units of 2^-24 per step
allow for a truncating accumulator, since the PTX documentation does not fix
the tensor core's internal rounding.

Here the accumulation is modelled in exact arithmetic plus one rounding per
block, to nearest even and toward zero, on random codes, on a large term with
tiny ones, and on blocks built to lose almost one ulp each.  The bound holds
in every case, and the last case shows it is nearly reached by a truncating
accumulator (and half reached when rounding to nearest), so it is not slack.
"""
import math

import numpy as np
import pytest

U = 2.0 ** -24


def round32(x: np.ndarray, mode: str) -> np.ndarray:
    r = x.astype(np.float32)                      # nearest even
    if mode == "rz":
        over = np.abs(r.astype(np.float64)) > np.abs(x)
        r = np.where(over, np.nextafter(r, np.float32(0.0)), r)
    return r


def accumulate(products: np.ndarray, mode: str) -> np.ndarray:
    """rows x K exact products -> fp32 accumulators, one rounding per block
    of 32 (the block sum itself exact)."""
    rows, K = products.shape
    acc = np.zeros(rows, dtype=np.float32)
    for j in range(0, K, 32):
        blk = products[:, j:j + 32].sum(axis=1)    # exact: multiples of 2^-18 below 2^35
        acc = round32(acc.astype(np.float64) + blk, mode)
    return acc


def bound(K, P):
    return (math.ceil(K / 32) + 1) * 2 * U * P


def e4m3_values(orc):
    v = np.array([orc.e4m3_bits_to_f64(b) for b in range(256)])
    return v[np.isfinite(v)]


@pytest.mark.parametrize("K", [32, 256, 3072, 12288])
@pytest.mark.parametrize("mode", ["rn", "rz"])
def test_bound_holds_on_random_codes(orc, K, mode):
    vals = e4m3_values(orc)
    rng = np.random.default_rng(K)
    a = rng.choice(vals, size=(64, K))
    w = rng.choice(vals, size=(64, K))
    p = a * w                                       # exact in fp64
    S = p.sum(axis=1)
    P = np.abs(p).sum(axis=1)
    err = np.abs(accumulate(p, mode).astype(np.float64) - S)
    assert np.all(err <= bound(K, P))


@pytest.mark.parametrize("mode", ["rn", "rz"])
def test_bound_holds_with_a_large_term_and_tiny_ones(mode):
    K = 12288
    p = np.full((1, K), 2.0 ** -18)                 # 2^-9 * 2^-9
    p[0, ::32] = 448.0 * 448.0
    S, P = p.sum(), np.abs(p).sum()
    assert abs(float(accumulate(p, mode)[0]) - S) <= bound(K, P)


def _losing_blocks(K, block_sum_units):
    """256 * 256 = 2^16 first (an ulp of 2^-7 = 2048 * 2^-18 at the
    accumulator), then blocks whose exact sum is `block_sum_units` * 2^-18:
    products of 2^-11 (2^-6 * 2^-5) and one of 120 * 2^-18 ((15 * 2^-9) *
    (8 * 2^-9)), the rest of the block zero."""
    p = np.zeros((1, K))
    n11, rest = divmod(block_sum_units - 120, 128)
    assert rest == 0 and n11 + 1 <= 32
    for j in range(K // 32):
        p[0, 32 * j:32 * j + n11] = 2.0 ** -11
        p[0, 32 * j + n11] = 120 * 2.0 ** -18
    p[0, 31] = 256.0 * 256.0                     # a zero slot of block 0
    return p


def test_bound_is_nearly_reached_by_a_truncating_accumulator():
    """Blocks just under one ulp (2040 of 2048): truncation drops every one,
    about 2^-23 |acc| per step, which is what the bound allows per step."""
    K = 12288
    p = _losing_blocks(K, 2040)
    S, P = p.sum(), np.abs(p).sum()
    err_rz = abs(float(accumulate(p, "rz")[0]) - S)
    err_rn = abs(float(accumulate(p, "rn")[0]) - S)
    assert 0.95 * bound(K, P) < err_rz <= bound(K, P)
    assert err_rn < 0.01 * bound(K, P)               # nearest rounding keeps each block


def test_bound_is_half_reached_when_rounding_to_nearest():
    """Blocks just under half an ulp (1016 of 2048): rounding to nearest
    drops every one."""
    K = 12288
    p = _losing_blocks(K, 1016)
    S, P = p.sum(), np.abs(p).sum()
    err_rn = abs(float(accumulate(p, "rn")[0]) - S)
    assert 0.45 * bound(K, P) < err_rn <= bound(K, P)
