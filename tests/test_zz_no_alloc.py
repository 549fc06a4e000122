"""The no-allocation GEMM entry point, checked against the regular one.

i8_gemm_dequant_bias_bf16_noalloc serves callers that cannot allocate device
memory when they call the layer: a plugin hosted by another runtime that
gives it no workspace, an application whose device memory all belongs to a
different allocator, or a latency-critical loop where cudaMalloc/cudaFree
(which may synchronize the device) are off limits.  Instead of a caller
workspace it uses a fixed 16 MiB scratch array inside the library.

This file is named so that pytest collects it last; it also passes when run
alone in a fresh process.
"""
import ctypes

import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import binding, inputs
from tests._util import assert_bf16_exact, gpu_bf16_bits

pytestmark = pytest.mark.gpu

VP = ctypes.c_void_p


def _prepared(M, N, K, seed):
    d = inputs.linear_inputs(inputs.LinearShape("na", M, K, N, seed=seed))
    x, w, b = (d[k].cuda() for k in ("x", "w", "bias"))
    aq, s_a = i8.quant_act_pertoken(x)
    wq, s_w = i8.quant_weight_perchannel(w)
    return aq, s_a, wq, s_w, b


def _noalloc(lib, aq, s_a, wq, s_w, b, y):
    M, K = aq.shape
    N = wq.shape[0]
    s = VP(torch.cuda.current_stream().cuda_stream)
    return lib.i8_gemm_dequant_bias_bf16_noalloc(
        VP(aq.data_ptr()), VP(s_a.data_ptr()), VP(wq.data_ptr()), VP(s_w.data_ptr()),
        VP(b.data_ptr()), M, N, K, VP(y.data_ptr()), y.stride(0), s)


def test_noalloc_matches_regular_entry_point_on_two_calls():
    lib = binding.load()
    i8.set_option("chunk_k", 1024)
    i8.set_option("force_splits", 0)
    # Two calls in a row, both on shapes that split K (so the fixed scratch is
    # used), the second one after the first has left its partials behind.
    for M, N, K, seed in ((16, 3072, 12288, 21), (2, 9216, 3072, 22)):
        assert i8.workspace_bytes(M, N, K) > 0
        aq, s_a, wq, s_w, b = _prepared(M, N, K, seed)
        y_ref = i8.gemm_dequant_bias_bf16(aq, s_a, wq, s_w, b)
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        assert _noalloc(lib, aq, s_a, wq, s_w, b, y) == 0
        i8.sync_check()
        assert_bf16_exact(gpu_bf16_bits(y), gpu_bf16_bits(y_ref), f"noalloc {M}x{N}x{K}")
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_noalloc_rejects_scratch_beyond_its_limit():
    lib = binding.load()
    M, N, K = 1024, 1024, 4096
    aq, s_a, wq, s_w, b = _prepared(M, N, K, 23)
    y = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    i8.set_option("force_splits", 16)      # 16 x 1024 x 1024 x 4 B = 64 MiB of partials
    try:
        assert i8.workspace_bytes(M, N, K) > 16 << 20
        assert _noalloc(lib, aq, s_a, wq, s_w, b, y) == 4   # I8_ERR_WORKSPACE
    finally:
        i8.set_option("force_splits", 0)
    i8.sync_check()
    assert not y.view(torch.int16).any()   # nothing was queued
