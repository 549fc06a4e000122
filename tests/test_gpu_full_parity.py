"""Whole-output parity at the full DiT sizes, every element against the oracle.

The pages' correctness claim is that the fused kernel's int32 accumulation is
bit-exact against torch._int_mm and its output matches the reference with
cosine 1.0 and no NaNs ("Realizing Native INT8 Compute for Diffusion
Transformers on Consumer GPUs", abstract).  Here every element of every
result is compared with the oracle at the full DiT layer sizes -- the QKV
projection at 768px (2560 x 3072 x 9216) and the MLP pair at 1024px, batch 2
(8704 x 3072 x 12288 up, 8704 x 12288 x 3072 down on GELU inputs):

* the exact routes (int8 codes widened on chip, on CTA pairs and on single
  CTAs, with int8 and with pre-widened weights; stream-K forced; the codes
  held as fp16 values): activation and weight codes and scales bit for bit,
  the whole int32 accumulator, and the whole bf16 output bit for bit;
* the E4M3 arm: codes and scales bit for bit, every fp32 accumulator within
  the derived rounding bound of the oracle's exact sum, and every bf16
  output equal to the oracle's epilogue of the GPU's accumulators and within
  tolerance of the exact path.

The oracle runs once per configuration (OpenMP over the host cores).
"""
import numpy as np
import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import inputs
from tests._util import assert_bf16_exact, gpu_bf16_bits, to_dev
from tests.test_gpu_e4m3 import acc_bound, _check_bf16

pytestmark = pytest.mark.gpu

FULL = [inputs.QKV_768, inputs.MLP_UP_1024, inputs.MLP_DOWN_1024]
OPTIONS = ("cta_pair", "stream_k")
ROWS_PER_CHUNK = 1024


@pytest.fixture
def saved_options():
    saved = {k: i8.get_option(k) for k in OPTIONS}
    yield
    for k, v in saved.items():
        i8.set_option(k, v)


def _f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("shape", FULL, ids=lambda s: s.name)
def test_full_size_exact_routes_every_element(orc, saved_options, shape):
    d = inputs.linear_inputs(shape)
    ref = orc.linear(inputs.bits(d["x"]), inputs.bits(d["w"]), inputs.bits(d["bias"]))
    x, w, b = to_dev(d["x"]), to_dev(d["w"]), to_dev(d["bias"])
    name = shape.name

    # codes and scales, bit for bit
    wq, s_w = i8.quant_weight_perchannel(w)
    aq, s_a = i8.quant_act_pertoken(x)
    i8.sync_check()
    assert np.array_equal(wq.cpu().numpy(), ref["wq"]), f"{name}: weight codes"
    assert np.array_equal(_f32_bits(s_w), ref["s_w"].view(np.uint32)), f"{name}: weight scales"
    assert np.array_equal(aq.cpu().numpy(), ref["aq"]), f"{name}: activation codes"
    assert np.array_equal(_f32_bits(s_a), ref["s_a"].view(np.uint32)), f"{name}: activation scales"

    # the whole int32 accumulator (the int8-code route's check path)
    c = i8.gemm_int32(aq, wq)
    i8.sync_check()
    assert np.array_equal(c.cpu().numpy(), ref["acc"]), f"{name}: int32 accumulators"
    del c

    want = ref["y"]
    # the fused layer on every exact route the table or an option can pick
    routes = [("table", {}), ("single CTA", {"cta_pair": 1}), ("CTA pairs", {"cta_pair": 2}),
              ("stream-K", {"cta_pair": 2, "stream_k": 2})]
    w16 = i8.widen_weight_codes(wq)
    for label, opts in routes:
        for k, v in opts.items():
            i8.set_option(k, v)
        y = i8.linear(x, wq, s_w, b)
        i8.sync_check()
        assert_bf16_exact(gpu_bf16_bits(y), want, f"{name} int8 codes, {label}")
        if label in ("table", "single CTA"):
            # the offline pre-widened weight copy (fp16 codes) on the same route
            y = i8.gemm_dequant_bias_bf16(aq, s_a, w16, s_w, b)
            i8.sync_check()
            assert_bf16_exact(gpu_bf16_bits(y), want, f"{name} pre-widened weights, {label}")
        del y
        for k in OPTIONS:
            i8.set_option(k, {"cta_pair": 0, "stream_k": 1}[k])

    # the same product with the codes held as fp16 values
    a16, s16 = i8.quant_act_pertoken_f16codes(x)
    i8.sync_check()
    assert np.array_equal(a16.cpu().numpy(), ref["aq"].astype(np.float16)), f"{name}: fp16 codes"
    assert np.array_equal(_f32_bits(s16), ref["s_a"].view(np.uint32))
    c16 = i8.gemm_int32_f16codes(a16, w16)
    i8.sync_check()
    assert np.array_equal(c16.cpu().numpy(), ref["acc"]), f"{name}: fp16-code int32 accumulators"
    del c16
    y = i8.linear_f16codes(x, w16, s_w, b)
    i8.sync_check()
    assert_bf16_exact(gpu_bf16_bits(y), want, f"{name} fp16-held codes")


@pytest.mark.parametrize("shape", FULL, ids=lambda s: s.name)
def test_full_size_e4m3_every_element(orc, shape):
    d = inputs.linear_inputs(shape)
    x = to_dev(d["x"])
    wq, s_w = i8.quant_weight_perchannel_e4m3(to_dev(d["w"]))
    aq, s_a = i8.quant_act_pertoken_e4m3(x)
    y = i8.gemm_e4m3_dequant_bias_bf16(aq, s_a, wq, s_w, to_dev(d["bias"]))
    c = i8.gemm_e4m3_f32(aq, wq)
    i8.sync_check()
    name = shape.name
    qo, so = orc.quant_rows_e4m3(inputs.bits(d["x"]))
    wo, swo = orc.quant_rows_e4m3(inputs.bits(d["w"]))
    a_codes = aq.view(torch.uint8).cpu().numpy()
    w_codes = wq.view(torch.uint8).cpu().numpy()
    assert np.array_equal(a_codes, qo), f"{name}: activation codes"
    assert np.array_equal(_f32_bits(s_a), so.view(np.uint32)), f"{name}: activation scales"
    assert np.array_equal(w_codes, wo), f"{name}: weight codes"
    assert np.array_equal(_f32_bits(s_w), swo.view(np.uint32)), f"{name}: weight scales"

    # the exact sum S of every accumulator from the oracle; the bound's
    # sum_k |a_k w_k| from a float64 matmul of the oracle's decoded |codes|
    # (non-negative terms: relative error below K * 2^-53, allowed for)
    exact = orc.gemm_e4m3_f64(qo, wo)
    table = torch.tensor([abs(orc.e4m3_bits_to_f64(v)) if v not in (0x7F, 0xFF) else 0.0
                          for v in range(256)], dtype=torch.float64)
    wabs = table[torch.from_numpy(wo.astype(np.int64))]
    got_all = c.cpu().numpy()
    y_all = gpu_bf16_bits(y)
    sa_np, sw_np = s_a.cpu().numpy(), s_w.cpu().numpy()
    bias_bits = inputs.bits(d["bias"])
    for r0 in range(0, shape.M, ROWS_PER_CHUNK):
        r1 = min(shape.M, r0 + ROWS_PER_CHUNK)
        aabs = table[torch.from_numpy(qo[r0:r1].astype(np.int64))]
        P = (aabs @ wabs.T).numpy() * (1 + 2.0 ** -40)
        got = got_all[r0:r1].astype(np.float64)
        assert np.isfinite(got).all(), f"{name}: NaN/Inf accumulators"
        err = np.abs(got - exact[r0:r1])
        bad = err > acc_bound(shape.K, P)
        assert not bad.any(), f"{name} rows {r0}..{r1}: {int(bad.sum())} accumulators beyond the bound"
        _check_bf16(orc, y_all[r0:r1], exact[r0:r1], P, got, sa_np[r0:r1], sw_np, bias_bits,
                    shape.K, f"{name} rows {r0}..{r1}")
