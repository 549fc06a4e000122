"""GPU parity of the per-row INT8 quantizer against the oracle: codes and
scales must be bit-identical (integer / byte work), on ragged, degenerate and
full-size inputs."""
import numpy as np
import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import inputs
from tests._util import to_dev

pytestmark = pytest.mark.gpu


def _compare(orc, x: torch.Tensor, fn=i8.quant_act_pertoken, what=""):
    q, s = fn(to_dev(x))
    torch.cuda.synchronize()
    q = q.cpu().numpy()
    s = s.cpu().numpy()
    oq, os_ = orc.quant_rows(inputs.bits(x))
    bad_s = np.flatnonzero(s.view(np.uint32) != os_.view(np.uint32))
    assert bad_s.size == 0, f"{what}: scale mismatch rows {bad_s[:8]} gpu {s[bad_s[:4]]} orc {os_[bad_s[:4]]}"
    bad = np.argwhere(q != oq)
    assert bad.size == 0, f"{what}: {len(bad)} code mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("M,K,dist,outl", [
    (64, 256, "normal", False),      # tiny config
    (1, 16, "normal", False),        # smallest K
    (7, 48, "normal", True),
    (129, 3072, "normal", True),     # DiT width, ragged M
    (33, 12288, "gelu", True),       # MLP down width: 4 warps per row
    (300, 1040, "normal", True),     # ragged vector tail inside a lane
    (17, 4096 + 16, "gelu", True),
    (5, 32768, "normal", True),      # longest row the register-resident kernel holds
    (9, 32768 + 16, "normal", True), # two-pass long-row kernel from here on
    (6, 131072, "gelu", True),       # maximum K
])
def test_quant_matches_oracle(orc, M, K, dist, outl):
    x = inputs.activations(M, K, torch.Generator().manual_seed(M * 7 + K), dist, outl)
    _compare(orc, x, what=f"{M}x{K}")


def test_quant_special_rows(orc):
    K = 64
    rows = []
    rows.append([0.0] * K)                                            # zero row
    rows.append([-0.0] * K)
    ties = [127.0, 2.5, -2.5, 3.5, -3.5, 0.5, -0.5, 1.5, -1.5, 126.5, -126.5, 125.5]
    rows.append(ties + [0.0] * (K - len(ties)))                      # scale 1: ties to even
    rows.append([63.5, 31.75, -0.25, 0.5, -63.5, 1.25, 0.75] + [0.25] * (K - 7))
    one = [0.0] * K
    one[37] = -3.0e-3
    rows.append(one)                                                  # single nonzero
    rows.append([-(i + 1) * 0.01 for i in range(K)])                  # all negative
    x = torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16)
    # subnormal rows (bf16 bit patterns), no flush to zero on either side
    sub = np.zeros((3, K), dtype=np.uint16)
    sub[0, :5] = [0x0001, 0x8003, 0x0005, 0x007F, 0x8040]
    sub[1, ::3] = 0x0002
    sub[2, :] = 0x00FF
    x = torch.cat([x, inputs.from_bits(sub)], dim=0)
    _compare(orc, x, what="special rows")


def test_quant_weight_perchannel_full_qkv(orc):
    d = inputs.linear_inputs(inputs.QKV_768)
    _compare(orc, d["w"], fn=i8.quant_weight_perchannel, what="W 9216x3072")


def test_quant_act_full_qkv(orc):
    d = inputs.linear_inputs(inputs.QKV_768)
    _compare(orc, d["x"], what="X 2560x3072")


def test_quant_act_full_mlp_down(orc):
    d = inputs.linear_inputs(inputs.MLP_DOWN_1024)
    _compare(orc, d["x"], what="X 8704x12288")


@pytest.mark.parametrize("rows", [1, 2, 4, 8])
@pytest.mark.parametrize("vpl", [1, 3, 6, 16])
def test_quant_launch_shapes_identical(orc, rows, vpl):
    """Every rows-per-CTA / vectors-per-lane launch shape gives the oracle's
    codes and scales (ragged M, ragged K tail, several warps per row)."""
    x = inputs.activations(45, 3072 + 48, torch.Generator().manual_seed(rows * 31 + vpl), "gelu", True)
    try:
        i8.set_option("quant_rows", rows)
        i8.set_option("quant_vpl", vpl)
        _compare(orc, x, what=f"rows{rows} vpl{vpl}")
    finally:
        i8.set_option("quant_rows", 0)
        i8.set_option("quant_vpl", 6)


def _all_bf16_up_to(amax_bits: int) -> np.ndarray:
    """Every finite bf16 bit pattern of magnitude <= the bf16 amax, both signs."""
    mags = np.arange(0, amax_bits + 1, dtype=np.uint32)
    return np.concatenate([mags, mags | 0x8000]).astype(np.uint16)


@pytest.mark.parametrize("fmt", ["int8", "f16codes"])
@pytest.mark.parametrize("amax", [127.0, 1.0, 300.0, 0.0173, 3.0e38, 1.0e-36])
def test_quant_every_bf16_input(orc, fmt, amax):
    """Exhaustive over the inputs: every bf16 value up to amax in magnitude,
    quantized with the scale amax / 127 (rows that start with amax), gives the
    oracle's code.  Covers the exact ties x / s = k + 1/2, quotients within a
    few fp32 ulps of a tie (where the reciprocal fast path must defer to the
    division), scale 1 (amax 127), and a subnormal scale (1e-36 / 127)."""
    K = 4096
    a_bits = int(np.array([amax], dtype=np.float32).view(np.uint32)[0] >> 16)
    vals = _all_bf16_up_to(a_bits)
    per_row = K - 1
    rows = -(-vals.size // per_row)
    xb = np.zeros((rows, K), dtype=np.uint16)
    xb[:, 0] = a_bits
    flat = np.zeros(rows * per_row, dtype=np.uint16)
    flat[:vals.size] = vals
    xb[:, 1:] = flat.reshape(rows, per_row)
    x = to_dev(inputs.from_bits(xb))
    if fmt == "int8":
        q, s = i8.quant_act_pertoken(x)
        got = q.cpu().numpy()
    else:
        q, s = i8.quant_act_pertoken_f16codes(x)
        got = q.cpu().float().numpy().astype(np.int8)
    i8.sync_check()
    qo, so = orc.quant_rows(xb)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    bad = np.argwhere(got != qo)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:4].tolist()}"
