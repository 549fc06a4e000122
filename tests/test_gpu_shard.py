"""GPU check of token sharding: every rank's slice, computed on its own, is
exactly the unsharded layer's rows.

The ranks are run one after another on the one GPU (they never wait on one
another).  On the exact routes (int8 codes, fp16-held codes) the slices must
equal the unsharded output bit for bit, whatever kernel each slice size
selects (the skinny weight-streaming kernel, split-K or the pair kernel); on
the E4M3 route the accumulation order may change with the slice's plan, so
each slice is held to the oracle's bound instead."""
import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import inputs
from w8a8_int8_quantized_i8_gb300.shard import linear_local, token_range
from tests._util import to_dev

pytestmark = pytest.mark.gpu


def _setup(M, N, K, codes):
    d = inputs.linear_inputs(inputs.LinearShape("t", M, K, N, seed=M + N, outliers=True))
    x, w, b = to_dev(d["x"]), to_dev(d["w"]), to_dev(d["bias"])
    if codes == "e4m3":
        wq, s_w = i8.quant_weight_perchannel_e4m3(w)
    else:
        wq, s_w = i8.quant_weight_perchannel(w)
        if codes == "f16codes":
            wq = i8.widen_weight_codes(wq)
    return d, x, wq, s_w, b


@pytest.mark.parametrize("codes", ["int8", "f16codes"])
@pytest.mark.parametrize("M,N,K,world", [(2561, 264, 400, 3), (10, 3072, 3072, 3),
                                         (2, 512, 256, 3), (1024, 1024, 4096, 8)])
def test_exact_slices_equal_unsharded(codes, M, N, K, world):
    d, x, wq, s_w, b = _setup(M, N, K, codes)
    full = linear_local(x, wq, s_w, b, 0, 1, codes=codes)
    parts = [linear_local(x, wq, s_w, b, r, world, codes=codes) for r in range(world)]
    i8.sync_check()
    assert [p.shape[0] for p in parts] == [token_range(M, r, world)[1] - token_range(M, r, world)[0]
                                           for r in range(world)]
    assert torch.equal(torch.cat(parts).view(torch.int16), full.view(torch.int16))


def test_e4m3_slices_within_oracle_bound(orc):
    """Each slice's codes and scales are the full run's rows bit for bit, and
    its accumulators and outputs meet the E4M3 arm's derived bound."""
    from tests.test_gpu_e4m3 import _check_acc, _check_bf16
    from tests._util import gpu_bf16_bits
    M, N, K, world = 515, 264, 1024, 4
    d, x, wq, s_w, b = _setup(M, N, K, "e4m3")
    aq_full, s_a_full = i8.quant_act_pertoken_e4m3(x)
    for r in range(world):
        m0, m1 = token_range(M, r, world)
        y = linear_local(x, wq, s_w, b, r, world, codes="e4m3")
        aq, s_a = i8.quant_act_pertoken_e4m3(x[m0:m1])
        c = i8.gemm_e4m3_f32(aq, wq)
        i8.sync_check()
        assert torch.equal(aq.view(torch.uint8), aq_full[m0:m1].view(torch.uint8))
        assert torch.equal(s_a, s_a_full[m0:m1])
        exact, P, got = _check_acc(orc, aq, wq, c, f"acc rank {r}")
        _check_bf16(orc, gpu_bf16_bits(y), exact, P, got, s_a.cpu().numpy(), s_w.cpu().numpy(),
                    inputs.bits(d["bias"]), K, f"rank {r}")
