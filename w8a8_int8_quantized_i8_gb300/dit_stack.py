"""A synthetic diffusion-transformer linear stack run through the W8A8 layer.

This is the workload of the pages' drop-in (the linear layers of a DiT,
"Realizing Native INT8 Compute for Diffusion Transformers on Consumer GPUs",
arXiv 2606.14598, abstract) with random-init weights, since the trained
Ideogram 4.0 weights are not available.  Per block, with M tokens of width
3072:

    h -> LN -> QKV (3072 -> 9216) -> V slice [6144:9216] (stands in for
    attention) -> LN -> out (3072 -> 3072) -> LN -> MLP up (3072 -> 12288)
    -> GELU -> MLP down (12288 -> 3072) -> LN -> next block

LN is a LayerNorm without affine parameters (eps 1e-6).  LN, GELU and the V
slice are torch glue between the layers and are not part of the measured
linear-layer path; every linear layer is per-token INT8 quantization of its
input followed by the fused int8 GEMM + dequant + bias (libi8).  Weights are
drawn with a seeded CUDA generator, ~N(0, 0.02), bias ~N(0, 0.01), and
quantized per output channel once (offline).
"""
from __future__ import annotations

import dataclasses

import torch

from . import binding as i8

WIDTH = 3072
LAYERS = (("qkv", 3072, 9216), ("out", 3072, 3072), ("up", 3072, 12288), ("down", 12288, 3072))


@dataclasses.dataclass
class Linear:
    wq: torch.Tensor      # int8 [N, K]
    s_w: torch.Tensor     # fp32 [N]
    bias: torch.Tensor    # bf16 [N]
    seed: int             # regenerates the bf16 weight for checks


def layer_weight(seed: int, N: int, K: int, device) -> tuple[torch.Tensor, torch.Tensor]:
    """The bf16 weight [N, K] and bias [N] of one layer (seeded, on `device`)."""
    g = torch.Generator(device=device).manual_seed(seed)
    w = (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    b = (torch.randn(N, generator=g, device=device, dtype=torch.float32) * 0.01).to(torch.bfloat16)
    return w, b


def build(blocks: int = 28, seed: int = 5, device="cuda") -> list[dict[str, Linear]]:
    """Quantized weights of `blocks` blocks (each layer's seed is derived from `seed`)."""
    stack = []
    for blk in range(blocks):
        layers = {}
        for li, (name, K, N) in enumerate(LAYERS):
            s = seed * 100003 + blk * 8 + li
            w, b = layer_weight(s, N, K, device)
            wq, s_w = i8.quant_weight_perchannel(w)
            del w
            layers[name] = Linear(wq, s_w, b, s)
        stack.append(layers)
    return stack


def layer_norm(x: torch.Tensor) -> torch.Tensor:
    return torch.nn.functional.layer_norm(x, (x.shape[-1],), eps=1e-6)


def forward(stack, h: torch.Tensor, record=None, timer=None) -> torch.Tensor:
    """Run the stack on h (bf16 [M, 3072]).  `record(blk, name, x, y)` sees
    every linear layer's input and output; `timer(begin: bool)` brackets each
    linear layer (quant + GEMM) for timing."""
    for blk, layers in enumerate(stack):
        x = layer_norm(h)
        for name in ("qkv", "out", "up", "down"):
            lin = layers[name]
            if timer:
                timer(True)
            y = i8.linear(x, lin.wq, lin.s_w, lin.bias)
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
