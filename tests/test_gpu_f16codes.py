"""GPU parity of the exact W8A8 path with the int8 codes held as fp16 values
(the quantizer's fp16-code output and offline-widened weights, fed to the
tensor core without on-chip widening).

Everything here is integer work decided in the same precision as the oracle,
so the bar is bit-exactness: the fp16 codes are the oracle's int8 codes, the
int32 accumulators equal the oracle's (also on adversarial +-127 operands
whose partial sums would leave fp32's exact range without the chunked
accumulation), and the bf16 outputs equal the oracle's and the int8-code
kernels' bit for bit."""
import numpy as np
import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import inputs
from tests._util import assert_bf16_exact, gpu_bf16_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(64, 256), (1, 16), (7, 48), (129, 3072), (33, 12288),
                                 (9, 32768 + 16), (2560, 3072)])
def test_quant_f16codes_are_the_int8_codes(orc, M, K):
    x = inputs.activations(M, K, torch.Generator().manual_seed(M + 2 * K))
    if M > 3:
        x[3] = 0.0
    q16, s = i8.quant_act_pertoken_f16codes(to_dev(x))
    i8.sync_check()
    qo, so = orc.quant_rows(inputs.bits(x))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    got = q16.cpu().float().numpy()
    assert np.array_equal(got, qo.astype(np.float32))
    if M > 3:
        assert (q16.cpu().view(torch.int16).numpy()[3] == 0).all()      # +0.0, not -0.0


SHAPES = [(64, 128, 256), (1, 8, 16), (7, 24, 48), (129, 136, 272), (256, 384, 1024),
          (300, 200, 1040), (1024, 1024, 4096), (513, 264, 400),
          # few tokens: the weight-streaming kernel with fp16-held codes on
          # both sides (cluster K splits); few tiles: the plan splits K
          # (exact int32 partials)
          (2, 9216, 3072), (16, 3072, 12288), (256, 3072, 3072), (32, 9216, 3072)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_int32_f16codes_matches_oracle(orc, M, N, K):
    a = inputs.random_int8(M, K, seed=M + K)
    w = inputs.random_int8(N, K, seed=N + 3 * K)
    c = i8.gemm_int32_f16codes(to_dev(a).half(), i8.widen_weight_codes(to_dev(w)))
    i8.sync_check()
    want = orc.gemm_s32(a.numpy(), w.numpy())
    bad = np.argwhere(c.cpu().numpy() != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("chunk_k", [64, 512, 1024])
def test_gemm_int32_f16codes_adversarial_exact(orc, chunk_k):
    """+-127 operands at K = 8192: exact only if the fp32 accumulator is
    restarted before its partial sums reach 2^24."""
    M, N, K = 260, 264, 8192
    g = torch.Generator().manual_seed(chunk_k)
    a = torch.full((M, K), 127, dtype=torch.int8)
    w = torch.full((N, K), 127, dtype=torch.int8)
    a[1:] *= (torch.randint(0, 2, (M - 1, K), generator=g, dtype=torch.int8) * 2 - 1)
    w[1:] *= (torch.randint(0, 2, (N - 1, K), generator=g, dtype=torch.int8) * 2 - 1)
    a[3] = -127
    i8.set_option("chunk_k", chunk_k)
    try:
        c = i8.gemm_int32_f16codes(to_dev(a).half(), to_dev(w).half())
        i8.sync_check()
    finally:
        i8.set_option("chunk_k", 1024)
    want = orc.gemm_s32(a.numpy(), w.numpy())
    assert np.array_equal(c.cpu().numpy(), want)
    assert c[0, 0].item() == 127 * 127 * K


@pytest.mark.parametrize("M,N,K,bias", [(64, 128, 256, True), (1, 8, 16, True), (7, 24, 48, False),
                                        (129, 136, 272, True), (300, 200, 1040, False),
                                        (16, 3072, 12288, True), (2, 9216, 3072, True)])
def test_linear_f16codes_matches_oracle_and_int8_path(orc, M, N, K, bias):
    shape = inputs.LinearShape("t", M, K, N, seed=M + N + K, outliers=K >= 256)
    d = inputs.linear_inputs(shape, with_bias=bias)
    wq, s_w = i8.quant_weight_perchannel(to_dev(d["w"]))
    b = None if d["bias"] is None else to_dev(d["bias"])
    y16 = i8.linear_f16codes(to_dev(d["x"]), i8.widen_weight_codes(wq), s_w, b)
    y8 = i8.linear(to_dev(d["x"]), wq, s_w, b)
    i8.sync_check()
    assert torch.equal(y16.view(torch.int16), y8.view(torch.int16))
    aq, s_a = orc.quant_rows(inputs.bits(d["x"]))
    wo, swo = orc.quant_rows(inputs.bits(d["w"]))
    want = orc.dequant_bias(orc.gemm_s32(aq, wo), s_a, swo,
                            None if d["bias"] is None else inputs.bits(d["bias"]))
    assert_bf16_exact(gpu_bf16_bits(y16), want, f"{M}x{N}x{K}")


def test_f16codes_workspace_errors():
    a = torch.zeros(32, 3072, dtype=torch.float16, device="cuda")
    w = torch.zeros(9216, 3072, dtype=torch.float16, device="cuda")
    need = i8.f16codes_workspace_bytes(32, 9216, 3072)
    assert need > 0
    with pytest.raises(i8.I8Error) as e:
        i8.gemm_int32_f16codes(a, w, workspace=torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 4
    i8.sync_check()


@pytest.mark.parametrize("splits", [2, 5, 16])
def test_f16codes_forced_splits_exact(orc, splits):
    """Any split count, also one whose K ranges do not line up with the
    accumulator restarts, gives the oracle's int32 sums and bf16 outputs."""
    M, N, K = 300, 520, 3072
    a = inputs.random_int8(M, K, seed=splits)
    w = inputs.random_int8(N, K, seed=splits + 1)
    shape = inputs.LinearShape("t", M, K, N, seed=splits, outliers=True)
    d = inputs.linear_inputs(shape)
    wq, s_w = i8.quant_weight_perchannel(to_dev(d["w"]))
    i8.set_option("force_splits", splits)
    try:
        assert i8.f16codes_workspace_bytes(M, N, K) > 0
        c = i8.gemm_int32_f16codes(to_dev(a).half(), to_dev(w).half())
        y = i8.linear_f16codes(to_dev(d["x"]), i8.widen_weight_codes(wq), s_w, to_dev(d["bias"]))
        i8.sync_check()
    finally:
        i8.set_option("force_splits", 0)
    assert np.array_equal(c.cpu().numpy(), orc.gemm_s32(a.numpy(), w.numpy()))
    want = orc.linear(inputs.bits(d["x"]), inputs.bits(d["w"]), inputs.bits(d["bias"]))["y"]
    assert_bf16_exact(gpu_bf16_bits(y), want, f"splits {splits}")


@pytest.mark.parametrize("M,N,K,splits", [(1, 200, 8192, 8), (7, 520, 3584, 7), (16, 136, 2560, 5)])
def test_f16codes_few_tokens_exact(orc, M, N, K, splits):
    """Few tokens with fp16-held codes on both sides take the weight-streaming
    kernel (forced cluster splits included): the oracle's int32 sums, no
    workspace."""
    a = inputs.random_int8(M, K, seed=M + 7)
    w = inputs.random_int8(N, K, seed=N + 9)
    i8.set_option("force_splits", splits)
    try:
        p = i8.plan_query(M, N, K, "f16codes")
        assert (p["kernel"], p["splits"], p["ws_bytes"]) == ("skinny", splits, 0)
        c = i8.gemm_int32_f16codes(to_dev(a).half(), to_dev(w).half())
        i8.sync_check()
    finally:
        i8.set_option("force_splits", 0)
    assert np.array_equal(c.cpu().numpy(), orc.gemm_s32(a.numpy(), w.numpy()))
