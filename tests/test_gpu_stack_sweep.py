"""Parity at the remaining DiT configurations: the 35-shape sweep (token
counts 1..16384 against the five DiT (K, N) pairs, skinny shapes exercising
split-K) and the synthetic 28-block linear stack at 1024px batch 2 (M = 8704)
with LayerNorm/GELU glue, every one of its 112 layers checked against the
oracle fed the GPU's own layer input.  Rows compared: all rows of a
few-token batch; otherwise one row of every 256-row M tile plus the first,
middle and last rows."""
import numpy as np
import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import dit_stack, inputs
from tests._util import assert_bf16_exact, gpu_bf16_bits

pytestmark = pytest.mark.gpu


def _rows(M):
    """Every row of a few-token batch; otherwise the first, middle and last
    eight rows plus one row of every 256-row M tile (the largest tile any
    kernel uses), at a position that moves from tile to tile."""
    if M <= 32:
        return np.arange(M)
    per_tile = np.array([256 * t + (97 * t + 13) % 256 for t in range(-(-M // 256))])
    return np.unique(np.concatenate([np.arange(8), np.arange(M // 2 - 4, M // 2 + 4),
                                     np.arange(M - 8, M), per_tile[per_tile < M]]))


def _oracle_rows(orc, x_bits_rows, w_bits, b_bits):
    aq, s_a = orc.quant_rows(x_bits_rows)
    wq, s_w = orc.quant_rows(w_bits)
    return orc.dequant_bias(orc.gemm_s32(aq, wq), s_a, s_w, b_bits)


@pytest.mark.parametrize("shape", inputs.sweep_shapes(), ids=lambda s: s.name)
def test_sweep_shape_every_m_tile(orc, shape):
    d = inputs.linear_inputs(shape)
    wq, s_w = i8.quant_weight_perchannel(d["w"].cuda())
    y = i8.linear(d["x"].cuda(), wq, s_w, d["bias"].cuda())
    i8.sync_check()
    rows = _rows(shape.M)
    want = _oracle_rows(orc, inputs.bits(d["x"][rows]), inputs.bits(d["w"]), inputs.bits(d["bias"]))
    assert_bf16_exact(gpu_bf16_bits(y)[rows], want, shape.name)
    # codes of the weights are bit-exact too
    assert np.array_equal(wq.cpu().numpy(), orc.quant_rows(inputs.bits(d["w"]))[0])


def test_dit_linear_stack_1024px_every_layer(orc):
    M = 8704
    stack = dit_stack.build(blocks=28, seed=5)
    h = inputs.activations(M, dit_stack.WIDTH, torch.Generator().manual_seed(5)).cuda()
    checks = {(blk, name) for blk in range(28) for name, _, _ in dit_stack.LAYERS}
    rows = _rows(M)
    seen = {}

    def record(blk, name, x, y):
        if (blk, name) in checks:
            seen[(blk, name)] = (x[rows].cpu(), y[rows].cpu())

    out = dit_stack.forward(stack, h, record=record)
    i8.sync_check()
    assert torch.isfinite(out.float()).all()
    assert set(seen) == checks
    for (blk, name), (x, y) in sorted(seen.items()):
        lin = stack[blk][name]
        K, N = lin.wq.shape[1], lin.wq.shape[0]
        w, b = dit_stack.layer_weight(lin.seed, N, K, "cuda")
        want = _oracle_rows(orc, inputs.bits(x), inputs.bits(w.cpu()), inputs.bits(b.cpu()))
        assert_bf16_exact(gpu_bf16_bits(y), want, f"block {blk} {name}")
