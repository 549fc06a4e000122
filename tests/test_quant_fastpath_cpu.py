"""The GPU quantizer's reciprocal fast path, modelled in fp32 on the CPU.

The quantizer's definition ("Realizing Native INT8 Compute for Diffusion
Transformers on Consumer GPUs", abstract: symmetric per-token INT8; the
oracle's reading: s = fl(amax / 127), q = round_half_even(fl(x / s))) asks
for one IEEE division per element.  The CUDA quantizer instead computes
t = fl(x * fl(1 / s)), rounds t with the 1.5 * 2^23 add, and takes the
division only for a vector where some |t - rint(t)| exceeds 1/2 - 2^-14
(or when s is subnormal).  Its claim: the fast codes always equal the
division's.

This test runs that decision rule in numpy fp32 (every step a single IEEE
operation, as on the GPU) against the oracle's division, for EVERY scale:
with s and 1/s both normal -- true for every bf16 amax whose scale is normal,
since s <= 2^121 -- scaling amax by 2^e scales s by 2^e and 1/s by 2^-e
exactly, so x / s, x * (1/s) and every rounding in between depend only on
amax's 8-bit significand and x's bits relative to it.  The 128 bf16
significands of amax in [1, 2), each with every bf16 x of magnitude up to
amax, are therefore all the cases there are.  The model also covers the
fused form that the kernel comment allows (x * fl(1/s) + 1.5 * 2^23 rounded
once), and the claim that the clamp to +-127 never binds on the fast path.
"""
import numpy as np

MAGIC = np.float32(12582912.0)               # 1.5 * 2^23
NEAR_TIE = np.float32(0.5) - np.float32(2.0 ** -14)


def _bf16_to_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _cases():
    """Rows [amax, x...]: each bf16 amax significand in [1, 2) with every
    bf16 value of magnitude below it, both signs."""
    rows = []
    for k in range(128):
        a_bits = np.uint16(0x3F80 + k)                    # (1 + k/128) * 2^0
        mags = np.arange(0, int(a_bits) + 1, dtype=np.uint16)
        xs = np.concatenate([mags, mags | np.uint16(0x8000)])
        rows.append((a_bits, xs))
    return rows


def test_fast_path_codes_equal_the_division_at_every_scale(orc):
    width = max(len(xs) for _, xs in _cases()) + 1
    fast_taken = 0
    total = 0
    for a_bits, xs in _cases():
        row = np.zeros((1, width), dtype=np.uint16)       # zero padding: code 0 on both sides
        row[0, 0] = a_bits
        row[0, 1:1 + len(xs)] = xs
        q_ref, s_ref = orc.quant_rows(row)
        amax = _bf16_to_f32(np.array([a_bits]))[0]
        s = np.float32(amax / np.float32(127.0))
        assert s.view(np.uint32) == s_ref[0].view(np.uint32)
        r = np.float32(np.float32(1.0) / s)
        x = _bf16_to_f32(row[0])
        t = (x * r).astype(np.float32)                     # fl(x * fl(1/s))
        y = (t + MAGIC).astype(np.float32)
        d = (t - (y - MAGIC).astype(np.float32)).astype(np.float32)
        code_fast = (y - MAGIC).astype(np.int64)
        # the fused form: the exact product (8 + 24 significant bits, exact in
        # fp64) plus the magic number (within 53 bits), rounded once to fp32
        y_fused = (x.astype(np.float64) * np.float64(r) + np.float64(MAGIC)).astype(np.float32)
        code_fused = (y_fused - MAGIC).astype(np.int64)
        fast = np.abs(d) <= NEAR_TIE
        ref = q_ref[0].astype(np.int64)
        assert np.array_equal(code_fast[fast], ref[fast]), a_bits
        assert np.array_equal(code_fused[fast], ref[fast]), a_bits
        assert np.abs(code_fast[fast]).max() <= 127       # no clamp needed on the fast path
        # the slow path is the plain division, which the oracle is
        fast_taken += int(fast.sum())
        total += fast.size
    # the near-tie band is narrow: almost every element takes the fast path
    assert fast_taken > 0.99 * total


def test_slow_path_cases_exist_and_are_true_near_ties(orc):
    """The rule defers only where the quotient is within a few fp32 ulps of a
    half-integer, and it defers every real tie (x / s a half-integer), where
    only the division gives the even code for certain.  Over all scales:
    about 4.2 M elements, a few hundred deferred, a few hundred exact ties."""
    deferred = 0
    exact_ties = 0
    for a_bits, xs in _cases():
        amax = _bf16_to_f32(np.array([a_bits]))[0]
        s = np.float32(amax / np.float32(127.0))
        r = np.float32(np.float32(1.0) / s)
        x = _bf16_to_f32(xs)
        t = (x * r).astype(np.float32)
        y = (t + MAGIC).astype(np.float32)
        d = (t - (y - MAGIC).astype(np.float32)).astype(np.float32)
        near = np.abs(d) > NEAR_TIE
        deferred += int(near.sum())
        q = (x.astype(np.float64) / np.float64(s))       # exact rational up to fp64 rounding
        frac = np.abs(q - np.trunc(q))
        ties = np.abs(frac - 0.5) == 0
        exact_ties += int(ties.sum())
        assert np.all(near[ties]), a_bits
        # every deferred element is within a few fp32 ulps of a half-integer
        assert np.all(np.abs(np.abs(q[near] - np.trunc(q[near])) - 0.5) < 2.0 ** -13)
    assert deferred > 0 and exact_ties > 0
