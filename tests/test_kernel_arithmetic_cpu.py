"""Arithmetic facts the exact int8 route rests on, checked exhaustively on the CPU.

sm_103a has no INT8 tensor-core MMA, so the int8 x int8 -> int32 product of
"Realizing Native INT8 Compute for Diffusion Transformers on Consumer GPUs"
(abstract) runs through the fp16 tensor pipe.  That is exact only because of
the facts below, each checked here for every case it covers.  The bit-level
steps are modelled from the documented semantics of the instructions the
kernels use (__byte_perm's byte selector, IEEE fp16 and fp32 arithmetic);
nothing here builds or runs device code.
"""
import numpy as np
import pytest


def byte_perm(x: int, y: int, s: int) -> int:
    """CUDA __byte_perm: result byte n is byte (s >> 4n) & 7 of the 8-byte
    value whose bytes 0-3 are x's and bytes 4-7 are y's."""
    src = (x & 0xFFFFFFFF) | ((y & 0xFFFFFFFF) << 32)
    out = 0
    for n in range(4):
        sel = (s >> (4 * n)) & 7
        out |= ((src >> (8 * sel)) & 0xFF) << (8 * n)
    return out


def s8x4_to_f16x4(w: int):
    """The widening of four int8 codes (one word) into four fp16 values, as
    the converters do it: x ^ 0x80 is x + 128 as an unsigned byte u; the fp16
    bit pattern 0x64uu is 1024 + u; an fp16 subtraction of 1152 (0x6480)
    leaves x."""
    u = w ^ 0x80808080
    a = byte_perm(u, 0x64646464, 0x4140)
    b = byte_perm(u, 0x64646464, 0x4342)
    halves = np.array([a & 0xFFFF, a >> 16, b & 0xFFFF, b >> 16], dtype=np.uint16).view(np.float16)
    return (halves - np.float16(1152.0)).astype(np.float16)


def test_every_int8_code_widens_exactly_at_every_byte_position():
    assert np.float16(1152.0).view(np.uint16) == 0x6480
    rng = np.random.default_rng(7)
    for code in range(-128, 128):
        for pos in range(4):
            for other in rng.integers(0, 1 << 32, size=8, dtype=np.uint64):
                w = int(other) & ~(0xFF << (8 * pos)) & 0xFFFFFFFF
                w |= (code & 0xFF) << (8 * pos)
                got = s8x4_to_f16x4(w)
                want = [int(np.int8(np.uint8((w >> (8 * i)) & 0xFF))) for i in range(4)]
                assert got.astype(np.int64).tolist() == want
                assert got[pos] == code


def test_fp16_holds_every_code_and_product_exactly():
    codes = np.arange(-128, 128)
    assert np.array_equal(codes.astype(np.float16).astype(np.int64), codes)
    p = np.outer(codes, codes)
    # each product of two fp16 integers of magnitude <= 128 is an integer
    # <= 2^14, exact in the fp32 accumulator
    assert np.array_equal(p.astype(np.float32).astype(np.int64), p)


def low_bytes4(b0, b1, b2, b3):
    """The quantizer's packing of four fp32 bit patterns' low bytes."""
    return byte_perm(byte_perm(b0, b1, 0x0040), byte_perm(b2, b3, 0x0040), 0x5410)


def test_code_packing_takes_the_low_byte_of_each_pattern_in_order():
    magic = int(np.float32(12582912.0).view(np.uint32))
    for q in range(-127, 128):
        pattern = int(np.float32(12582912.0 + q).view(np.uint32))
        assert pattern == magic + q                   # the ulp at 1.5 * 2^23 is 1
        assert pattern & 0xFF == q & 0xFF
    rng = np.random.default_rng(3)
    for _ in range(2000):
        qs = rng.integers(-127, 128, size=4)
        pats = [int(np.float32(12582912.0 + int(q)).view(np.uint32)) for q in qs]
        word = low_bytes4(*pats)
        got = [int(np.int8(np.uint8((word >> (8 * i)) & 0xFF))) for i in range(4)]
        assert got == qs.tolist()


@pytest.mark.parametrize("chunk", list(range(64, 1025, 64)))
def test_fp32_chunk_accumulation_is_exact(chunk):
    """Every chunk length the GEMM allows keeps each partial sum of int8
    products inside fp32's exact integer range, in any order of summation:
    |partial| <= 127^2 * chunk < 2^24 for the quantizers' codes, and
    <= 128^2 * chunk <= 2^24 even with -128 codes."""
    assert 127 * 127 * chunk < 1 << 24
    assert 128 * 128 * chunk <= 1 << 24
    rng = np.random.default_rng(chunk)
    worst = [np.full(chunk, 127 * 127), np.full(chunk, -127 * 127), np.full(chunk, 128 * 128),
             rng.integers(-128, 128, chunk) * rng.integers(-128, 128, chunk)]
    for p in worst:
        acc = np.float32(0.0)
        for v in p:                               # sequential fp32 adds, each rounded
            acc = np.float32(acc + np.float32(v))
        assert int(acc) == int(p.sum())


def test_int32_totals_fit_for_every_allowed_k():
    """The drained chunk sums are added in int32: 127^2 * K < 2^31 for every
    K <= 131072 (the library's limit); with -128 codes only K = 131072 with
    every product (-128)^2 reaches 2^31."""
    assert 127 * 127 * 131072 < 1 << 31
    assert 127 * 127 * 133144 < 1 << 31 <= 127 * 127 * 133145
    assert 128 * 128 * 131071 < 1 << 31 == 128 * 128 * 131072
