"""The seeded input recipe the oracle and the GPU share (no GPU needed):
same seed -> same bytes, the outlier structure, the value distributions and
the layer shapes the workloads name."""
import numpy as np
import pytest
import torch

from w8a8_int8_quantized_i8_gb300 import inputs


def test_same_seed_same_bytes_other_seed_other_bytes():
    a = inputs.linear_inputs(inputs.TINY)
    b = inputs.linear_inputs(inputs.TINY)
    for k in ("x", "w", "bias"):
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16))
    c = inputs.linear_inputs(inputs.LinearShape("t", 64, 256, 128, seed=1, outliers=False))
    assert not torch.equal(a["x"].view(torch.int16), c["x"].view(torch.int16))
    # bits() and from_bits() are inverse
    assert torch.equal(inputs.from_bits(inputs.bits(a["x"])).view(torch.int16), a["x"].view(torch.int16))


@pytest.mark.parametrize("K", [256, 3072, 12288])
def test_outlier_channels(K):
    """round(0.01 K) whole channels are scaled by 20, the rest are N(0, 1)."""
    M = 512
    x = inputs.activations(M, K, torch.Generator().manual_seed(K), "normal", True).float()
    col_std = x.std(dim=0)
    loud = torch.nonzero(col_std > 8.0).flatten()
    assert loud.numel() == int(round(0.01 * K))
    assert float(col_std[loud].mean()) == pytest.approx(20.0, rel=0.15)
    quiet = torch.ones(K, dtype=torch.bool)
    quiet[loud] = False
    assert float(col_std[quiet].mean()) == pytest.approx(1.0, rel=0.05)
    # without outliers no channel stands out
    y = inputs.activations(M, K, torch.Generator().manual_seed(K), "normal", False).float()
    assert float(y.std(dim=0).max()) < 2.0


def test_gelu_inputs_and_weight_scales():
    d = inputs.linear_inputs(inputs.LinearShape("t", 1024, 1024, 256, seed=5, x_dist="gelu",
                                                outliers=False))
    x = d["x"].float()
    # GELU(N(0,1)): bounded below by min GELU ~ -0.17, mean ~ 0.28
    assert float(x.min()) > -0.18
    assert float(x.mean()) == pytest.approx(0.2821, abs=0.01)
    assert float(d["w"].float().std()) == pytest.approx(0.02, rel=0.05)
    assert float(d["bias"].float().std()) == pytest.approx(0.01, rel=0.2)


def test_workload_shapes():
    assert (inputs.QKV_768.M, inputs.QKV_768.K, inputs.QKV_768.N) == (2304 + 256, 3072, 9216)
    assert (inputs.MLP_UP_1024.M, inputs.MLP_UP_1024.K, inputs.MLP_UP_1024.N) == (2 * (4096 + 256), 3072, 12288)
    assert (inputs.MLP_DOWN_1024.K, inputs.MLP_DOWN_1024.N, inputs.MLP_DOWN_1024.x_dist) == (12288, 3072, "gelu")
    sweep = inputs.sweep_shapes()
    assert len(sweep) == 35
    assert {s.M for s in sweep} == {1, 2, 16, 256, 1024, 4096, 16384}
    assert {(s.K, s.N) for s in sweep} == {(3072, 9216), (3072, 3072), (3072, 12288), (12288, 3072),
                                           (3072, 18432)}
    assert all(s.x_dist == ("gelu" if s.K == 12288 else "normal") for s in sweep)
    assert (inputs.TINY.seed, inputs.TINY.outliers) == (0, False)
