"""Token (M) sharding of the W8A8 linear layer over several GPUs.

The layer shards without any exchange along the token dimension: the
activation scales are per token ("Realizing Native INT8 Compute for Diffusion
Transformers on Consumer GPUs", arXiv 2606.14598, abstract: per-token
activation and per-channel weight quantization), so a row's codes, its
accumulators and its output depend on that row and the weights only.  Each
rank holds the full quantized weights and computes a contiguous slice of the
rows; the slices are exactly the rows the unsharded layer would produce.  A
collective is needed only when one rank wants the whole output (gather_rows).

Everything here is host-side bookkeeping around the library's calls.
"""
from __future__ import annotations

import torch

from . import binding as i8


def token_range(M: int, rank: int, world: int) -> tuple[int, int]:
    """Rows [m0, m1) of rank `rank`: contiguous, balanced (the first M % world
    ranks take one row more), covering 0..M exactly once."""
    if world < 1 or not 0 <= rank < world or M < 0:
        raise ValueError("bad rank/world/M")
    base, extra = divmod(M, world)
    m0 = rank * base + min(rank, extra)
    return m0, m0 + base + (1 if rank < extra else 0)


def linear_local(x_full: torch.Tensor, wq, s_w, bias, rank: int, world: int,
                 codes: str = "int8", out=None, workspace=None) -> torch.Tensor:
    """This rank's rows of the layer: quantize and multiply x_full[m0:m1].

    ``codes`` picks the route: "int8" (wq int8), "f16codes" (wq widened) or
    "e4m3" (wq E4M3).  Returns the bf16 [m1 - m0, N] slice.
    """
    m0, m1 = token_range(x_full.shape[0], rank, world)
    x = x_full[m0:m1]
    if m1 == m0:
        return torch.empty((0, wq.shape[0]), dtype=torch.bfloat16, device=x_full.device)
    if codes == "int8":
        return i8.linear(x, wq, s_w, bias, out=out, workspace=workspace)
    if codes == "f16codes":
        return i8.linear_f16codes(x, wq, s_w, bias, out=out, workspace=workspace)
    if codes == "e4m3":
        return i8.linear_e4m3(x, wq, s_w, bias, out=out, workspace=workspace)
    raise ValueError(f"unknown codes {codes!r}")


def gather_rows(y_local: torch.Tensor, M: int, rank: int, world: int, group=None) -> torch.Tensor:
    """All ranks' slices stacked into the full [M, N] output on every rank
    (torch.distributed all_gather; slices are padded to the largest and
    trimmed, since M need not divide by the world size)."""
    import torch.distributed as dist
    N = y_local.shape[1]
    rows = max(token_range(M, r, world)[1] - token_range(M, r, world)[0] for r in range(world))
    pad = torch.zeros((rows, N), dtype=y_local.dtype, device=y_local.device)
    pad[: y_local.shape[0]] = y_local
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    out = []
    for r in range(world):
        m0, m1 = token_range(M, r, world)
        out.append(parts[r][: m1 - m0])
    return torch.cat(out, dim=0)
