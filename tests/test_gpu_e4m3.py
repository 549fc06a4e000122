"""GPU parity of the E4M3 (FP8) arm against the oracle.

* Codes and scales: bit-exact (both sides decide each code from the same
  correctly rounded fp32 quotient x / s).
* fp32 accumulators: the tensor core adds in fp32 in an unspecified order, so
  they are checked against the oracle's exact fp64 sum S with the bound
      |acc - S| <= (ceil(K / 32) + 17) * 2 * 2^-24 * sum_k |a_k w_k|,
  i.e. at most one rounding (allowed 2 ulp, since the tensor core's adder
  rounding mode is not documented) per K = 32 MMA step, per addition of a
  K split's partial in the fix-up (at most 16 splits), and the final one.
* bf16 outputs: bit-identical to the oracle's epilogue applied to the GPU's
  own fp32 accumulators (the epilogue steps are the same fp32 operations);
  and against the oracle's exact path within one bf16 ulp plus the
  accumulator bound scaled by s_a * s_w, with cosine >= 0.99999 and no
  NaN/Inf.
"""
import math

import numpy as np
import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import inputs
from tests._util import ABS_TOL, COS_MIN, REL_TOL, bits_to_f64, gpu_bf16_bits, to_dev

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def _codes(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.uint8).cpu().numpy()


def acc_bound(K: int, P: np.ndarray) -> np.ndarray:
    # one rounding per K = 32 MMA step, plus up to 16 for a K split's
    # partials being added in the fix-up, plus the final one
    return (math.ceil(K / 32) + 17) * 2 * U * P


def _check_acc(orc, aq, wq, c, what=""):
    a, w = _codes(aq), _codes(wq)
    K = a.shape[1]
    exact = orc.gemm_e4m3_f64(a, w)
    P = orc.gemm_e4m3_f64(a, w, absval=True)
    got = c.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: NaN/Inf"
    err = np.abs(got - exact)
    bad = err > acc_bound(K, P)
    assert not bad.any(), (f"{what}: {int(bad.sum())} accumulators beyond the bound, worst "
                           f"{(err / np.maximum(P, 1e-300)).max() / U:.2f} u * P")
    return exact, P, got


def _check_bf16(orc, y_bits, exact, P, got_acc, s_a, s_w, bias_bits, K, what=""):
    # (1) the GPU epilogue is the oracle's epilogue on the GPU's accumulators
    want_own = orc.dequant_bias_f64acc(got_acc, s_a, s_w, bias_bits)
    diff = np.argwhere(y_bits != want_own)
    assert diff.size == 0, f"{what}: {len(diff)} bf16 outputs differ from the oracle epilogue"
    # (2) within tolerance of the exact path
    want = orc.dequant_bias_f64acc(exact, s_a, s_w, bias_bits)
    g = bits_to_f64(y_bits)
    w = bits_to_f64(want)
    assert np.isfinite(g).all()
    scale = s_a.astype(np.float64)[:, None] * s_w.astype(np.float64)[None, :]
    tol = REL_TOL * np.abs(w) + ABS_TOL + scale * acc_bound(K, P) * (1 + 2.0 ** -20)
    bad = np.abs(g - w) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs beyond tolerance"
    denom = np.linalg.norm(g) * np.linalg.norm(w)
    if denom > 0:
        assert float((g * w).sum() / denom) >= COS_MIN


# ----------------------------------------------------------------- quantizer
@pytest.mark.parametrize("R,K", [(64, 256), (1, 16), (7, 48), (129, 3072), (300, 12288),
                                 (33, 131072), (2560, 3072)])
def test_quant_e4m3_bit_exact(orc, R, K):
    x = inputs.activations(R, K, torch.Generator().manual_seed(R + K))
    if R > 3:
        x[3] = 0.0                                        # zero row
        x[2] = x[2].float().mul(1e-36).to(torch.bfloat16)  # tiny row: subnormal scale
    q, s = i8.quant_act_pertoken_e4m3(to_dev(x))
    i8.sync_check()
    qo, so = orc.quant_rows_e4m3(inputs.bits(x))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    bad = np.argwhere(_codes(q) != qo)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:4].tolist()}"


def test_quant_e4m3_weights_and_special_rows(orc):
    w = inputs.random_bf16(40, 512, seed=8, std=0.02)
    w[0] = 0.0
    w[1, :] = -0.0
    w[2, 7] = 448.0                   # scale 1: codes are E4M3(x) itself
    w[2, :7] = 3.0
    w[3] = torch.linspace(-1, 1, 512).to(torch.bfloat16)
    q, s = i8.quant_weight_perchannel_e4m3(to_dev(w))
    i8.sync_check()
    qo, so = orc.quant_rows_e4m3(inputs.bits(w))
    assert np.array_equal(_codes(q), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert s[0].item() == 0.0 and s[1].item() == 0.0
    assert (_codes(q)[:2] == 0).all()


def _all_bf16_up_to(amax_bits: int) -> np.ndarray:
    """Every finite bf16 bit pattern of magnitude <= the bf16 amax, both signs."""
    mags = np.arange(0, amax_bits + 1, dtype=np.uint32)
    return np.concatenate([mags, mags | 0x8000]).astype(np.uint16)


@pytest.mark.parametrize("amax", [1.0, 300.0, 0.0173, 3.0e38, 5.0e-37, 448.0])
def test_quant_e4m3_every_bf16_input(orc, amax):
    """Exhaustive over the inputs: every bf16 value up to amax in magnitude,
    quantized with the scale amax / 448 (rows that start with amax), gives
    the oracle's code.  Covers exact E4M3 ties, values within a few fp32 ulps
    of a rounding boundary (where the fast path must defer to the division),
    saturation at 448, a subnormal scale (5e-37 / 448) and scale 1."""
    K = 4096
    a_bits = int(np.array([amax], dtype=np.float32).view(np.uint32)[0] >> 16)
    amax_bf16 = float(np.array([a_bits << 16], dtype=np.uint32).view(np.float32)[0])
    vals = _all_bf16_up_to(a_bits)
    per_row = K - 1
    rows = -(-vals.size // per_row)
    xb = np.zeros((rows, K), dtype=np.uint16)
    xb[:, 0] = a_bits                                  # every row's absmax is amax
    flat = np.zeros(rows * per_row, dtype=np.uint16)
    flat[:vals.size] = vals
    xb[:, 1:] = flat.reshape(rows, per_row)
    x = inputs.from_bits(xb)
    q, s = i8.quant_act_pertoken_e4m3(to_dev(x))
    i8.sync_check()
    qo, so = orc.quant_rows_e4m3(xb)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert float(so[0]) == np.float32(amax_bf16) / np.float32(448.0)
    bad = np.argwhere(_codes(q) != qo)
    assert bad.size == 0, f"amax {amax_bf16}: {len(bad)} codes differ, first {bad[:4].tolist()}"


# ----------------------------------------------------------------- GEMM
GEMM_SHAPES = [(64, 128, 256), (1, 8, 16), (7, 24, 48), (129, 136, 272), (300, 520, 1040),
               (256, 256, 3072), (200, 304, 12288), (513, 264, 400),
               # few tokens (the weight-streaming kernel: E4M3 m16n8k32 MMAs,
               # cluster K splits summed in a fixed order) and few tiles (the
               # cost model splits K for the last one: fp32 partials + ordered
               # fix-up)
               (16, 3072, 3072), (256, 9216, 3072), (1, 3072, 12288), (2, 18432, 3072),
               (32, 3072, 3072)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_e4m3_f32_within_bound(orc, M, N, K):
    x = inputs.activations(M, K, torch.Generator().manual_seed(M + K))
    w = inputs.random_bf16(N, K, seed=N + 3 * K, std=0.02)
    aq, _ = i8.quant_act_pertoken_e4m3(to_dev(x))
    wq, _ = i8.quant_weight_perchannel_e4m3(to_dev(w))
    c = i8.gemm_e4m3_f32(aq, wq)
    i8.sync_check()
    _check_acc(orc, aq, wq, c, f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(32, 3072, 3072), (64, 3072, 12288)])
def test_gemm_e4m3_split_k_is_deterministic(M, N, K):
    assert i8.e4m3_workspace_bytes(M, N, K) > 0          # these shapes split K
    a = torch.randint(0, 0x7E, (M, K), dtype=torch.uint8, device="cuda")
    w = torch.randint(0, 0x7E, (N, K), dtype=torch.uint8, device="cuda") | 0x80
    c1 = i8.gemm_e4m3_f32(a, w)
    ws = torch.full((i8.e4m3_workspace_bytes(M, N, K),), 0xFF, dtype=torch.uint8, device="cuda")
    c2 = i8.gemm_e4m3_f32(a, w, workspace=ws)            # garbage in the workspace is fine
    i8.sync_check()
    assert torch.equal(c1.view(torch.int32), c2.view(torch.int32))
    with pytest.raises(i8.I8Error) as e:
        i8.gemm_e4m3_f32(a, w, workspace=ws[:-16])
    assert e.value.status == 4


@pytest.mark.parametrize("M,N,K,splits", [(1, 3072, 12288, 0), (5, 520, 3584, 7), (16, 136, 2560, 5),
                                           (3, 200, 8192, 8)])
def test_gemm_e4m3_few_tokens(orc, M, N, K, splits):
    """Few tokens take the weight-streaming kernel: no workspace, the
    accumulators within the bound, the same bits on every call (the K splits
    of a cluster are summed in a fixed order), and bf16 outputs equal to the
    oracle's epilogue of those accumulators."""
    shape = inputs.LinearShape("t", M, K, N, seed=M + K, outliers=True)
    d = inputs.linear_inputs(shape)
    aq, s_a = i8.quant_act_pertoken_e4m3(to_dev(d["x"]))
    wq, s_w = i8.quant_weight_perchannel_e4m3(to_dev(d["w"]))
    i8.set_option("force_splits", splits)
    try:
        p = i8.plan_query(M, N, K, "e4m3")
        assert p["kernel"] == "skinny" and p["ws_bytes"] == 0
        if splits:
            assert p["splits"] == splits
        assert i8.e4m3_workspace_bytes(M, N, K) == 0
        c = i8.gemm_e4m3_f32(aq, wq)
        c2 = i8.gemm_e4m3_f32(aq, wq)
        y = i8.gemm_e4m3_dequant_bias_bf16(aq, s_a, wq, s_w, to_dev(d["bias"]))
        i8.sync_check()
    finally:
        i8.set_option("force_splits", 0)
    assert torch.equal(c.view(torch.int32), c2.view(torch.int32))
    exact, P, got = _check_acc(orc, aq, wq, c, f"{M}x{N}x{K} splits {splits}")
    _check_bf16(orc, gpu_bf16_bits(y), exact, P, got, s_a.cpu().numpy(), s_w.cpu().numpy(),
                inputs.bits(d["bias"]), K, f"{M}x{N}x{K} splits {splits}")


def test_gemm_e4m3_closed_forms(orc):
    # all ones: every partial sum is a small integer, exact in fp32
    M, N, K = 260, 272, 4096
    ones = torch.full((M, K), 0x38, dtype=torch.uint8, device="cuda")
    onesw = torch.full((N, K), 0x38, dtype=torch.uint8, device="cuda")
    c = i8.gemm_e4m3_f32(ones, onesw)
    i8.sync_check()
    assert (c == K).all()
    # +-448 extremes: partial sums are multiples of 448^2 = 49 * 2^12 below 2^28, exact in fp32
    big = torch.full((M, 1024), 0x7E, dtype=torch.uint8, device="cuda")
    neg = torch.full((N, 1024), 0xFE, dtype=torch.uint8, device="cuda")
    c = i8.gemm_e4m3_f32(big, neg)
    i8.sync_check()
    assert (c == -448.0 * 448.0 * 1024).all()
    # identity weights reproduce the decoded rows (catches a transposed operand)
    a = torch.randint(0, 0x7E, (300, 256), dtype=torch.uint8)
    eye = torch.where(torch.eye(256, dtype=torch.bool), 0x38, 0x00).to(torch.uint8)
    c = i8.gemm_e4m3_f32(to_dev(a), to_dev(eye))
    i8.sync_check()
    want = a.view(torch.float8_e4m3fn).to(torch.float32)
    assert torch.equal(c.cpu(), want)


def test_gemm_e4m3_mixed_magnitudes_within_bound(orc):
    # large and tiny terms in every K = 32 block: the accumulator rounding the
    # bound allows for is exercised (the tiny terms are each half an ulp)
    M, N, K = 256, 256, 4096
    a = torch.full((M, K), 0x7E, dtype=torch.uint8)
    a[:, 1::2] = 0x01
    w = torch.full((N, K), 0x38, dtype=torch.uint8)
    c = i8.gemm_e4m3_f32(to_dev(a), to_dev(w))
    i8.sync_check()
    _check_acc(orc, a, w, c, "mixed")


@pytest.mark.parametrize("M,N,K,bias", [(64, 128, 256, True), (1, 8, 16, True), (7, 24, 48, False),
                                        (129, 136, 272, True), (300, 520, 1040, False),
                                        (16, 3072, 3072, True), (256, 9216, 3072, True),
                                        (2, 12288, 3072, False)])
def test_linear_e4m3_matches_oracle(orc, M, N, K, bias):
    shape = inputs.LinearShape("t", M, K, N, seed=M + N + K, outliers=K >= 256)
    d = inputs.linear_inputs(shape, with_bias=bias)
    aq, s_a = i8.quant_act_pertoken_e4m3(to_dev(d["x"]))
    wq, s_w = i8.quant_weight_perchannel_e4m3(to_dev(d["w"]))
    b = None if d["bias"] is None else to_dev(d["bias"])
    y = i8.gemm_e4m3_dequant_bias_bf16(aq, s_a, wq, s_w, b)
    c = i8.gemm_e4m3_f32(aq, wq)
    i8.sync_check()
    exact, P, got = _check_acc(orc, aq, wq, c, "acc")
    bb = None if d["bias"] is None else inputs.bits(d["bias"])
    _check_bf16(orc, gpu_bf16_bits(y), exact, P, got, s_a.cpu().numpy(), s_w.cpu().numpy(), bb,
                K, f"{M}x{N}x{K}")
    # the whole path through the public call gives the same bits
    y2 = i8.linear_e4m3(to_dev(d["x"]), wq, s_w, b)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_e4m3_zero_rows_give_bias():
    M, N, K = 5, 64, 128
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[2] = 1.0
    w = inputs.random_bf16(N, K, seed=3, std=0.02)
    b = inputs.random_bf16(1, N, seed=4, std=0.5)[0]
    wq, s_w = i8.quant_weight_perchannel_e4m3(to_dev(w))
    y = i8.linear_e4m3(to_dev(x), wq, s_w, to_dev(b))
    i8.sync_check()
    yb = gpu_bf16_bits(y)
    for r in (0, 1, 3, 4):
        assert np.array_equal(yb[r], inputs.bits(b))


def test_e4m3_error_paths():
    a = torch.zeros(64, 128, dtype=torch.uint8, device="cuda")
    raw = torch.zeros(64 * 128 + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(i8.I8Error) as e:
        i8.gemm_e4m3_f32(raw[1:1 + 64 * 128].view(64, 128), a)
    assert e.value.status == 2
    with pytest.raises(i8.I8Error) as e:
        i8.gemm_e4m3_f32(torch.zeros(4, 24, dtype=torch.uint8, device="cuda"),
                         torch.zeros(8, 24, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 3
    i8.sync_check()


@pytest.mark.parametrize("splits", [2, 5, 16])
def test_gemm_e4m3_forced_splits_within_bound(orc, splits):
    """Any split count (uneven K ranges included) keeps the accumulators
    within the bound and gives the same bf16 outputs as the oracle's
    epilogue on those accumulators."""
    M, N, K = 300, 520, 3072
    shape = inputs.LinearShape("t", M, K, N, seed=splits, outliers=True)
    d = inputs.linear_inputs(shape)
    aq, s_a = i8.quant_act_pertoken_e4m3(to_dev(d["x"]))
    wq, s_w = i8.quant_weight_perchannel_e4m3(to_dev(d["w"]))
    i8.set_option("force_splits", splits)
    try:
        assert i8.e4m3_workspace_bytes(M, N, K) > 0
        c = i8.gemm_e4m3_f32(aq, wq)
        y = i8.gemm_e4m3_dequant_bias_bf16(aq, s_a, wq, s_w, to_dev(d["bias"]))
        i8.sync_check()
    finally:
        i8.set_option("force_splits", 0)
    exact, P, got = _check_acc(orc, aq, wq, c, f"splits {splits}")
    _check_bf16(orc, gpu_bf16_bits(y), exact, P, got, s_a.cpu().numpy(), s_w.cpu().numpy(),
                inputs.bits(d["bias"]), K, f"splits {splits}")
