"""Seeded synthetic inputs shaped like diffusion-transformer linear layers.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no quantization, no GEMM, no epilogue), so both the CUDA
path and the CPU oracle can consume the same bytes.

Recipe (one ``torch.Generator`` on the CPU per call, fp32 draws cast to bf16,
draw order fixed as X, outlier-channel permutation, W, bias):

* X ~ N(0, 1), or GELU(N(0, 1)) (erf form) for the input of an MLP
  down-projection; when outliers are on, ``round(0.01 * K)`` channels picked by
  ``randperm(K)`` are scaled by 20 -- the activation-outlier structure that
  motivates per-token scales.
* W ~ N(0, 0.02) in the ``[out, in]`` = ``[N, K]`` layout.
* bias ~ N(0, 0.01).

The layer shapes are those of a 3072-wide DiT (QKV 3072->9216, attention out
3072->3072, MLP 3072->12288->3072, adaLN modulation 3072->18432) at 768px and
1024px token counts.  The pages benchmark Ideogram 4.0's own layers, whose
weights and prompts are not available, so these synthetic tensors stand in.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class LinearShape:
    name: str
    M: int
    K: int
    N: int
    seed: int
    x_dist: str = "normal"      # "normal" or "gelu"
    outliers: bool = True


# The tiny case the oracle finishes instantly (seed 0, no outliers).
TINY = LinearShape("tiny_M64_K256_N128", 64, 256, 128, seed=0, outliers=False)
# DiT QKV projection at 768px, batch 1: 2304 image + 256 text tokens.
QKV_768 = LinearShape("dit_qkv_768px_M2560_K3072_N9216", 2560, 3072, 9216, seed=2)
# DiT MLP pair at 1024px, batch 2 with CFG: 2 x (4096 + 256) tokens.
MLP_UP_1024 = LinearShape("dit_mlp_up_1024px_M8704_K3072_N12288", 8704, 3072, 12288, seed=3)
MLP_DOWN_1024 = LinearShape("dit_mlp_down_1024px_M8704_K12288_N3072", 8704, 12288, 3072,
                            seed=3, x_dist="gelu")

SWEEP_M = (1, 2, 16, 256, 1024, 4096, 16384)
SWEEP_KN = ((3072, 9216), (3072, 3072), (3072, 12288), (12288, 3072), (3072, 18432))


def sweep_shapes():
    """The 35-shape sweep: every token count against every DiT (K, N) pair."""
    out = []
    for K, N in SWEEP_KN:
        for M in SWEEP_M:
            out.append(LinearShape(f"sweep_M{M}_K{K}_N{N}", M, K, N, seed=4,
                                   x_dist="gelu" if K == 12288 else "normal"))
    return out


def _gelu_erf(x: torch.Tensor) -> torch.Tensor:
    return torch.nn.functional.gelu(x, approximate="none")


def activations(M: int, K: int, g: torch.Generator, x_dist: str = "normal",
                outliers: bool = True) -> torch.Tensor:
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    if x_dist == "gelu":
        x = _gelu_erf(x)
    elif x_dist != "normal":
        raise ValueError(x_dist)
    n_out = int(round(0.01 * K))
    idx = torch.randperm(K, generator=g)[:n_out]
    if outliers and n_out > 0:
        x[:, idx] *= 20.0
    return x.to(torch.bfloat16)


def linear_inputs(shape: LinearShape, with_bias: bool = True):
    """``dict(x=[M,K] bf16, w=[N,K] bf16, bias=[N] bf16 or None)`` on the CPU."""
    g = torch.Generator().manual_seed(shape.seed)
    x = activations(shape.M, shape.K, g, shape.x_dist, shape.outliers)
    w = (torch.randn(shape.N, shape.K, generator=g, dtype=torch.float32) * 0.02)
    w = w.to(torch.bfloat16)
    b = (torch.randn(shape.N, generator=g, dtype=torch.float32) * 0.01).to(torch.bfloat16)
    return dict(x=x, w=w, bias=b if with_bias else None)


def random_bf16(rows: int, cols: int, seed: int, std: float = 1.0) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def random_int8(rows: int, cols: int, seed: int, lo: int = -127, hi: int = 127) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (rows, cols), generator=g, dtype=torch.int32).to(torch.int8)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 CPU tensor -> numpy uint16 bit patterns."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected bf16")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
