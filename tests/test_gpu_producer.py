"""GPU parity of the fused producer-quantizers (LayerNorm or GELU, then the
per-token quantizer, in one kernel) against the oracle.

* The bf16 producer output y (the kernel's optional output).  GELU: equal to
  the oracle's fp64 value rounded once, everywhere (the kernel reads a table
  of exactly those values).  LayerNorm: within one bf16 step of it (plus the
  fp32 mean's rounding bound, which matters only where y is near 0), and
  equal almost everywhere (the kernel reduces in fp32, so values within fp32
  noise of a rounding midpoint may round the other way).
* Codes and scales: bit-exact against the oracle's quantizer applied to the
  GPU's own y (the integer decision is taken from the same bf16 row).
* Asking for y does not change the codes.
* The fused DiT stack: every checked layer's output is bit-identical to the
  oracle's linear layer fed the layer's bf16 input.
"""
import numpy as np
import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import dit_stack, inputs
from tests._util import assert_bf16_exact, bits_to_f64, gpu_bf16_bits, to_dev

pytestmark = pytest.mark.gpu


def _codes(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).cpu().numpy()
    if t.dtype == torch.float16:                 # fp16-held int8 codes
        return t.cpu().float().numpy().astype(np.int8)
    return t.cpu().numpy()


def _run(op, x, fmt, want_y):
    if op == "layernorm":
        return i8.layernorm_quant_act_pertoken(x, eps=1e-6, fmt=fmt, want_y=want_y)
    return i8.gelu_quant_act_pertoken(x, fmt=fmt, want_y=want_y)


def _check(orc, op, x_cpu, fmt, min_exact=0.999):
    x = to_dev(x_cpu)
    q, s, y = _run(op, x, fmt, True)
    q2, s2 = _run(op, x, fmt, False)
    i8.sync_check()
    yb = gpu_bf16_bits(y)
    xb = inputs.bits(x_cpu)
    y_ref = orc.layernorm_rows(xb, 1e-6) if op == "layernorm" else orc.gelu_rows(xb)
    g, w = bits_to_f64(yb), bits_to_f64(y_ref)
    assert np.isfinite(g).all()
    # within one bf16 step: |g - w| <= 2^-7 |w| (+ the subnormal spacing).
    # For the LayerNorm add the error of the fp32 mean, which the kernel's
    # reduction bounds by 2^-24 * sum_k |x_k| (one rounding per addition,
    # doubled for the reduction order), scaled by 1/sqrt(var + eps): it
    # dominates where x is close to the mean and y close to 0.
    tol = 2.0 ** -7 * np.abs(w) + 2.0 ** -133
    if op == "layernorm":
        xf = bits_to_f64(xb)
        rstd = 1.0 / np.sqrt(xf.var(axis=1) + 1e-6)
        tol = tol + (rstd * 2.0 * 2.0 ** -24 * np.abs(xf).sum(axis=1))[:, None]
    bad = np.abs(g - w) > tol
    assert not bad.any(), f"{int(bad.sum())} producer outputs beyond one bf16 step"
    frac = float((yb == y_ref).mean())
    if op == "gelu":
        # the GELU producer reads a table of the fp64 value rounded once: the
        # oracle's definition, so every output is equal
        min_exact = 1.0
    assert frac >= min_exact, f"only {frac:.5f} of the producer outputs equal the oracle's"
    # codes and scales from the GPU's own bf16 row, bit for bit
    qo, so = orc.quant_rows_e4m3(yb) if fmt == "e4m3" else orc.quant_rows(yb)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    bad = np.argwhere(_codes(q) != qo)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:4].tolist()}"
    # the optional output does not change the codes
    assert torch.equal(q.view(torch.uint8), q2.view(torch.uint8)) and torch.equal(s, s2)
    if fmt == "f16codes":                         # exact integers, +0.0 for zero
        qf = q.cpu().float().numpy()
        assert np.array_equal(qf, np.round(qf)) and not np.signbit(qf[qf == 0]).any()
    return frac


@pytest.mark.parametrize("fmt", ["int8", "e4m3", "f16codes"])
@pytest.mark.parametrize("op", ["layernorm", "gelu"])
@pytest.mark.parametrize("M,K", [(64, 256), (7, 48), (1, 16), (129, 3072), (33, 12288),
                                 (5, 32768), (2560, 3072)])
def test_producer_quant_matches_oracle(orc, op, fmt, M, K):
    g = torch.Generator().manual_seed(M * 3 + K)
    x = inputs.activations(M, K, g, "normal")
    if op == "layernorm":
        x = (x.float() * 0.5 + 0.25).to(torch.bfloat16)        # a nonzero mean to remove
    _check(orc, op, x, fmt)


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
def test_layernorm_special_rows(orc, fmt):
    K = 512
    rows = torch.randn(6, K, generator=torch.Generator().manual_seed(1))
    rows[0] = 0.0                        # zero row: y = 0, scale 0, codes 0
    rows[1] = 3.5                        # constant row: x - mu = 0
    rows[2] = rows[2] * 1e-3 + 100.0     # large mean, small spread
    rows[3, ::2] = 1.0
    rows[3, 1::2] = -1.0                 # mean 0, variance 1: y = +-1
    x = rows.to(torch.bfloat16)
    _check(orc, "layernorm", x, fmt, min_exact=0.99)
    q, s = i8.layernorm_quant_act_pertoken(to_dev(x), fmt=fmt)
    i8.sync_check()
    assert s[0].item() == 0.0 and s[1].item() == 0.0
    assert (_codes(q)[:2] == 0).all()


def test_gelu_every_bf16_input_matches_oracle(orc):
    """All 65536 bf16 patterns (finite ones) through the GELU producer: each
    output is the oracle's correctly rounded GELU."""
    pats = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        keep = np.isfinite((pats.astype(np.uint32) << 16).view(np.float32))
    pats = pats[keep]
    pats = pats[: len(pats) // 256 * 256].reshape(-1, 256)
    x = inputs.from_bits(pats)
    _, _, y = i8.gelu_quant_act_pertoken(to_dev(x), want_y=True)
    i8.sync_check()
    assert np.array_equal(gpu_bf16_bits(y), orc.gelu_rows(pats))


def test_producer_strided_input_and_errors(orc):
    # a column slice of a wider matrix (the V third of a QKV output), no copy
    wide = inputs.activations(96, 9216, torch.Generator().manual_seed(3))
    xw = to_dev(wide)
    q, s, y = i8.layernorm_quant_act_pertoken(xw[:, 6144:9216], want_y=True)
    qc, sc, yc = i8.layernorm_quant_act_pertoken(xw[:, 6144:9216].contiguous(), want_y=True)
    i8.sync_check()
    assert torch.equal(q, qc) and torch.equal(s, sc) and torch.equal(y.view(torch.int16), yc.view(torch.int16))
    with pytest.raises(i8.I8Error) as e:
        i8.gelu_quant_act_pertoken(torch.zeros(4, 32768 + 16, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == 3
    with pytest.raises(ValueError):
        i8.gelu_quant_act_pertoken(torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda"), fmt="nf4")


def _rows(M):
    """First, middle and last eight rows plus one row of every 256-row M tile."""
    per_tile = np.array([256 * t + (97 * t + 13) % 256 for t in range(-(-M // 256))])
    return np.unique(np.concatenate([np.arange(8), np.arange(M // 2 - 4, M // 2 + 4),
                                     np.arange(M - 8, M), per_tile[per_tile < M]]))


def test_fused_dit_stack_every_layer_every_m_tile(orc):
    M = 8704
    stack = dit_stack.build(blocks=4, seed=5)
    h = inputs.activations(M, dit_stack.WIDTH, torch.Generator().manual_seed(5)).cuda()
    rows = _rows(M)
    seen = {}

    def record(blk, name, x, y):
        seen[(blk, name)] = (x[rows].cpu(), y[rows].cpu())

    out = dit_stack.forward(stack, h, record=record, fused=True)
    ref = dit_stack.forward(stack, h, fused=False)
    i8.sync_check()
    assert torch.isfinite(out.float()).all()
    # the fused stack tracks the unfused one (their LayerNorms round in
    # different fp32 orders, so the two differ by a few bf16 steps at most)
    cos = torch.nn.functional.cosine_similarity(out.float().flatten(), ref.float().flatten(), dim=0)
    assert cos.item() > 0.999
    for (blk, name), (x, y) in sorted(seen.items()):
        lin = stack[blk][name]
        K, N = lin.wq.shape[1], lin.wq.shape[0]
        w, b = dit_stack.layer_weight(lin.seed, N, K, "cuda")
        aq, s_a = orc.quant_rows(inputs.bits(x))
        wq, s_w = orc.quant_rows(inputs.bits(w.cpu()))
        want = orc.dequant_bias(orc.gemm_s32(aq, wq), s_a, s_w, inputs.bits(b.cpu()))
        assert_bf16_exact(gpu_bf16_bits(y), want, f"block {blk} {name}")


@pytest.mark.parametrize("fused", [False, True])
def test_f16codes_stack_is_bit_identical_to_int8_stack(fused):
    """The fp16-held codes change the storage, not the arithmetic: two blocks of
    the DiT stack give the same bits through either path."""
    M = 1024
    h = inputs.activations(M, dit_stack.WIDTH, torch.Generator().manual_seed(9)).cuda()
    s8 = dit_stack.build(blocks=2, seed=7, fmt="int8")
    s16 = dit_stack.build(blocks=2, seed=7, fmt="f16codes")
    o8 = dit_stack.forward(s8, h, fused=fused)
    o16 = dit_stack.forward(s16, h, fused=fused)
    i8.sync_check()
    assert torch.equal(o8.view(torch.int16), o16.view(torch.int16))
