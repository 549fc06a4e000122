"""Shared helpers for the parity tests: moving seeded inputs to the GPU and
comparing results with the oracle.  No method arithmetic lives here."""
import numpy as np
import torch


# bf16 parity bar: |gpu - oracle| <= 2^-7 * |oracle| + 1e-6 per element (one
# bf16 ulp), cosine >= 0.99999, no NaN/Inf.
REL_TOL = 2.0 ** -7
ABS_TOL = 1e-6
COS_MIN = 0.99999


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gpu_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_bf16_close(got_bits: np.ndarray, want_bits: np.ndarray, what: str = ""):
    g = bits_to_f64(got_bits)
    w = bits_to_f64(want_bits)
    assert np.isfinite(g).all(), f"{what}: NaN/Inf in GPU output"
    err = np.abs(g - w)
    bad = err > REL_TOL * np.abs(w) + ABS_TOL
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond 1 bf16 ulp; "
                           f"worst {err.max():.3g}")
    denom = np.linalg.norm(g) * np.linalg.norm(w)
    if denom > 0:
        cos = float((g * w).sum() / denom)
        assert cos >= COS_MIN, f"{what}: cosine {cos}"
    return float((got_bits == want_bits).mean())


def finite_bits(b: np.ndarray) -> bool:
    """No NaN or Inf among bf16 bit patterns (exponent field all ones)."""
    return not ((b & 0x7F80) == 0x7F80).any()


def assert_bf16_exact(got_bits: np.ndarray, want_bits: np.ndarray, what: str = ""):
    """Bit-identical bf16: the GPU epilogue takes the oracle's fp32 steps in
    the same order with the same rounding.  Equal, finite bits are within any
    tolerance with cosine 1; otherwise the 1-ulp check runs first so a
    failure says whether the difference is a rounding step or a real error."""
    assert got_bits.shape == want_bits.shape, f"{what}: shape {got_bits.shape} != {want_bits.shape}"
    if np.array_equal(got_bits, want_bits):
        assert finite_bits(got_bits), f"{what}: NaN/Inf in GPU output"
        return
    assert_bf16_close(got_bits, want_bits, what)
    bad = np.argwhere(got_bits != want_bits)
    assert bad.size == 0, (f"{what}: {len(bad)} of {got_bits.size} elements differ by one "
                           f"rounding step, first {bad[:4].tolist()}")


def to_dev(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().to("cuda")


def int8_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()
