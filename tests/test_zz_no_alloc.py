"""The no-allocation GEMM entry point, checked against the oracle.

i8_gemm_dequant_bias_bf16_noalloc serves callers that cannot allocate device
memory when they call the layer: a plugin hosted by another runtime that
gives it no workspace, an application whose device memory all belongs to a
different allocator, or a latency-critical loop where cudaMalloc/cudaFree
(which may synchronize the device) are off limits.  Instead of a caller
workspace it uses a fixed 16 MiB scratch array inside the library, and caps
its launch plan to that size.

Every route through the array is covered: the tiled kernels' split-K
partials, a shape whose regular plan needs more than 16 MiB (so the capped
plan splits K fewer times), and the stream-K schedule, whose arrival words
stay behind in the array between calls; and the few-token kernel, whose K
splits meet in distributed shared memory and use none of it.  Each shape is
called twice in a row and both results must equal the oracle's bit for
bit.

This file is named so that pytest collects it last; it also passes when run
alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import w8a8_int8_quantized_i8_gb300 as i8
from w8a8_int8_quantized_i8_gb300 import binding, inputs
from tests._util import assert_bf16_exact, gpu_bf16_bits

pytestmark = pytest.mark.gpu

VP = ctypes.c_void_p
STATIC_BYTES = 16 << 20
OPTIONS = ("chunk_k", "force_splits", "stream_k", "cta_pair")


@pytest.fixture
def saved_options():
    saved = {k: i8.get_option(k) for k in OPTIONS}
    yield
    for k, v in saved.items():
        i8.set_option(k, v)


def _case(orc, M, N, K, seed):
    d = inputs.linear_inputs(inputs.LinearShape("na", M, K, N, seed=seed))
    x, w, b = (d[k].cuda() for k in ("x", "w", "bias"))
    aq, s_a = i8.quant_act_pertoken(x)
    wq, s_w = i8.quant_weight_perchannel(w)
    want = orc.linear(inputs.bits(d["x"]), inputs.bits(d["w"]), inputs.bits(d["bias"]))["y"]
    return (aq, s_a, wq, s_w, b), want


def _noalloc(lib, aq, s_a, wq, s_w, b, y):
    M, K = aq.shape
    N = wq.shape[0]
    s = VP(torch.cuda.current_stream().cuda_stream)
    return lib.i8_gemm_dequant_bias_bf16_noalloc(
        VP(aq.data_ptr()), VP(s_a.data_ptr()), VP(wq.data_ptr()), VP(s_w.data_ptr()),
        VP(b.data_ptr()), M, N, K, VP(y.data_ptr()), y.stride(0), s)


def _twice_against_oracle(orc, lib, M, N, K, seed, what):
    args, want = _case(orc, M, N, K, seed)
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(lib, *args, y) == 0
        i8.sync_check()
        assert_bf16_exact(gpu_bf16_bits(y), want, f"noalloc {what} {M}x{N}x{K} call {call}")


@pytest.mark.parametrize("M,N,K,seed,route", [
    (32, 3072, 12288, 21, "tiled split-K"),
    (2, 3072, 12288, 22, "few-token cluster split-K"),
    (256, 3072, 3072, 24, "split-K capped to the array"),
    (256, 9216, 3072, 26, "split-K capped to none"),
])
def test_noalloc_matches_oracle_on_two_calls(orc, saved_options, M, N, K, seed, route):
    lib = binding.load()
    i8.set_option("chunk_k", 1024)
    i8.set_option("force_splits", 0)
    p = i8.plan_query(M, N, K, "int8")
    capped = i8.plan_query(M, N, K, "int8", ws_cap=STATIC_BYTES)
    assert capped["ws_bytes"] <= STATIC_BYTES
    if route.startswith("few-token"):
        # K splits, and no scratch at all
        assert p["kernel"] == "skinny" and p["splits"] > 1 and p["ws_bytes"] == 0
        assert capped == p
    else:
        assert p["ws_bytes"] > 0                 # the regular plan needs scratch
    if route.startswith("split-K capped"):
        # the regular plan's partials outgrow the array: fewer splits
        assert p["ws_bytes"] > STATIC_BYTES and capped["splits"] < p["splits"]
    if route in ("tiled split-K", "split-K capped to the array"):
        assert capped["ws_bytes"] > 0           # the array is used
    _twice_against_oracle(orc, lib, M, N, K, seed, route)


def test_noalloc_stream_k_on_two_calls(orc, saved_options):
    """Stream-K through the array: its arrival words stay behind between
    calls and only their per-launch tag makes the second call start afresh."""
    lib = binding.load()
    i8.set_option("cta_pair", 2)
    i8.set_option("stream_k", 2)
    M, N, K = 256, 768, 4096            # 3 tiles of 32 K blocks on up to 24 pairs
    p = i8.plan_query(M, N, K, "int8", ws_cap=STATIC_BYTES)
    assert p["kernel"] == "pair_stream_k" and 0 < p["ws_bytes"] <= STATIC_BYTES
    _twice_against_oracle(orc, lib, M, N, K, 25, "stream-K")


def test_noalloc_rejects_scratch_beyond_its_limit(saved_options):
    lib = binding.load()
    M, N, K = 1024, 1024, 4096
    d = inputs.linear_inputs(inputs.LinearShape("na", M, K, N, seed=23))
    aq, s_a = i8.quant_act_pertoken(d["x"].cuda())
    wq, s_w = i8.quant_weight_perchannel(d["w"].cuda())
    b = d["bias"].cuda()
    y = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    i8.set_option("force_splits", 16)      # 16 x 1024 x 1024 x 4 B = 64 MiB of partials
    assert i8.workspace_bytes(M, N, K) > STATIC_BYTES
    assert _noalloc(lib, aq, s_a, wq, s_w, b, y) == 4   # I8_ERR_WORKSPACE
    i8.sync_check()
    assert not y.view(torch.int16).any()   # nothing was queued
    assert np.all(np.isfinite(y.float().cpu().numpy()))
