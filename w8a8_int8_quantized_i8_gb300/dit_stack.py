"""A synthetic diffusion-transformer linear stack run through the W8A8 layer.

This is the workload of the pages' drop-in (the linear layers of a DiT,
"Realizing Native INT8 Compute for Diffusion Transformers on Consumer GPUs",
arXiv 2606.14598, abstract) with random-init weights, since the trained
Ideogram 4.0 weights are not available.  Per block, with M tokens of width
3072:

    h -> LN -> QKV (3072 -> 9216) -> V slice [6144:9216] (stands in for
    attention) -> LN -> out (3072 -> 3072) -> LN -> MLP up (3072 -> 12288)
    -> GELU -> MLP down (12288 -> 3072) -> LN -> next block

LN is a LayerNorm without affine parameters (eps 1e-6).  Two ways to run it:

* unfused (default): LN, GELU and the V slice are torch glue between the
  layers; every linear layer is the per-token quantizer of its bf16 input
  followed by the fused GEMM + dequant + bias (libi8);
* fused: the LayerNorm in front of QKV / out / up and the GELU in front of
  down run inside libi8's producer kernels, which write the next layer's codes
  directly (the bf16 layer input is never written); only the block-output LN
  and the V slice (a strided view, no copy) stay outside.

``fmt`` picks the codes: "int8" (the exact int8 path), "f16codes" (the same
exact path with the codes held as fp16 values, weights widened offline) or
"e4m3" (the FP8 arm).  Weights are drawn with a seeded CUDA generator, ~N(0, 0.02), bias
~N(0, 0.01), and quantized per output channel once (offline).
"""
from __future__ import annotations

import dataclasses

import torch

from . import binding as i8

WIDTH = 3072
LAYERS = (("qkv", 3072, 9216), ("out", 3072, 3072), ("up", 3072, 12288), ("down", 12288, 3072))


@dataclasses.dataclass
class Linear:
    wq: torch.Tensor      # int8 or E4M3 codes [N, K]
    s_w: torch.Tensor     # fp32 [N]
    bias: torch.Tensor    # bf16 [N]
    seed: int             # regenerates the bf16 weight for checks
    fmt: str = "int8"


def layer_weight(seed: int, N: int, K: int, device) -> tuple[torch.Tensor, torch.Tensor]:
    """The bf16 weight [N, K] and bias [N] of one layer (seeded, on `device`)."""
    g = torch.Generator(device=device).manual_seed(seed)
    w = (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    b = (torch.randn(N, generator=g, device=device, dtype=torch.float32) * 0.01).to(torch.bfloat16)
    return w, b


def build(blocks: int = 28, seed: int = 5, device="cuda", fmt: str = "int8") -> list[dict[str, Linear]]:
    """Quantized weights of `blocks` blocks (each layer's seed is derived from `seed`)."""
    quant = i8.quant_weight_perchannel_e4m3 if fmt == "e4m3" else i8.quant_weight_perchannel
    stack = []
    for blk in range(blocks):
        layers = {}
        for li, (name, K, N) in enumerate(LAYERS):
            s = seed * 100003 + blk * 8 + li
            w, b = layer_weight(s, N, K, device)
            wq, s_w = quant(w)
            if fmt == "f16codes":
                wq = i8.widen_weight_codes(wq)
            del w
            layers[name] = Linear(wq, s_w, b, s, fmt)
        stack.append(layers)
    return stack


def layer_norm(x: torch.Tensor) -> torch.Tensor:
    return torch.nn.functional.layer_norm(x, (x.shape[-1],), eps=1e-6)


def _gemm(lin: Linear, aq, s_a):
    if lin.fmt == "int8":
        return i8.gemm_dequant_bias_bf16(aq, s_a, lin.wq, lin.s_w, lin.bias)
    if lin.fmt == "f16codes":
        return i8.gemm_dequant_bias_bf16_f16codes(aq, s_a, lin.wq, lin.s_w, lin.bias)
    return i8.gemm_e4m3_dequant_bias_bf16(aq, s_a, lin.wq, lin.s_w, lin.bias)


def forward(stack, h: torch.Tensor, record=None, timer=None, fused: bool = False) -> torch.Tensor:
    """Run the stack on h (bf16 [M, 3072]).  `record(blk, name, x, y)` sees
    every linear layer's bf16 input and output; `timer(begin: bool)` brackets
    each linear layer (its quantizer -- fused with the LN / GELU in front of
    it when `fused` -- and the GEMM) for timing."""
    if fused:
        return _forward_fused(stack, h, record, timer)
    for blk, layers in enumerate(stack):
        x = layer_norm(h)
        for name in ("qkv", "out", "up", "down"):
            lin = layers[name]
            if timer:
                timer(True)
            if lin.fmt == "int8":
                y = i8.linear(x, lin.wq, lin.s_w, lin.bias)
            elif lin.fmt == "f16codes":
                y = i8.linear_f16codes(x, lin.wq, lin.s_w, lin.bias)
            else:
                y = i8.linear_e4m3(x, lin.wq, lin.s_w, lin.bias)
            if timer:
                timer(False)
            if record:
                record(blk, name, x, y)
            if name == "qkv":
                x = layer_norm(y[:, 2 * WIDTH:3 * WIDTH].contiguous())
            elif name == "out":
                x = layer_norm(y)
            elif name == "up":
                x = torch.nn.functional.gelu(y, approximate="none")
            else:
                h = layer_norm(y)
    return h


def _forward_fused(stack, h, record, timer):
    want_y = record is not None
    for blk, layers in enumerate(stack):
        src, op = h, "layernorm"
        for name in ("qkv", "out", "up", "down"):
            lin = layers[name]
            if timer:
                timer(True)
            if op == "layernorm":
                r = i8.layernorm_quant_act_pertoken(src, eps=1e-6, fmt=lin.fmt, want_y=want_y)
            else:
                r = i8.gelu_quant_act_pertoken(src, fmt=lin.fmt, want_y=want_y)
            y = _gemm(lin, r[0], r[1])
            if timer:
                timer(False)
            if record:
                record(blk, name, r[2], y)
            if name == "qkv":
                src, op = y[:, 2 * WIDTH:3 * WIDTH], "layernorm"   # strided view, no copy
            elif name == "out":
                src, op = y, "layernorm"
            elif name == "up":
                src, op = y, "gelu"
            else:
                h = layer_norm(y)
    return h
