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
