"""Token sharding on CPU: the row split and the gather, with two gloo ranks.

Each rank computes its rows of the layer with the oracle (the product path
needs a GPU); the gathered result must equal the unsharded oracle bit for bit,
which holds because per-token quantization makes every output row a function
of its own input row and the weights only.  No GPU is involved.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from w8a8_int8_quantized_i8_gb300.shard import token_range


@pytest.mark.parametrize("M,world", [(0, 1), (1, 1), (5, 2), (2560, 2), (2561, 3), (3, 8), (4096, 8)])
def test_token_range_partitions_rows(M, world):
    spans = [token_range(M, r, world) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == M
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0                                   # contiguous, no overlap, no gap
    sizes = [m1 - m0 for m0, m1 in spans]
    assert min(sizes) >= 0 and max(sizes) - min(sizes) <= 1
    assert sizes == sorted(sizes, reverse=True)           # the longer slices come first


def test_token_range_rejects_bad_arguments():
    for args in [(4, 2, 2), (4, -1, 2), (4, 0, 0), (-1, 0, 1)]:
        with pytest.raises(ValueError):
            token_range(*args)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, M, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import oracle
    from w8a8_int8_quantized_i8_gb300 import inputs
    from w8a8_int8_quantized_i8_gb300.shard import gather_rows
    dist.init_process_group("gloo", rank=rank, world_size=world)
    d = inputs.linear_inputs(inputs.LinearShape("t", M, 96, 40, seed=11, outliers=True))
    m0, m1 = token_range(M, rank, world)
    if m1 > m0:
        y = oracle.linear(inputs.bits(d["x"][m0:m1]), inputs.bits(d["w"]), inputs.bits(d["bias"]))["y"]
    else:                                    # this rank owns no tokens
        y = np.zeros((0, 40), dtype=np.uint16)
    y_full = gather_rows(torch.from_numpy(y.astype(np.int32)), M, rank, world)     # bf16 bits
    q.put((rank, y_full.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("M,world", [(7, 3), (64, 2), (2, 3)])
def test_gathered_slices_equal_unsharded_layer(orc, M, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, M, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    from w8a8_int8_quantized_i8_gb300 import inputs
    d = inputs.linear_inputs(inputs.LinearShape("t", M, 96, 40, seed=11, outliers=True))
    want = orc.linear(inputs.bits(d["x"]), inputs.bits(d["w"]), inputs.bits(d["bias"]))["y"]
    for rank, got in out:
        assert got.shape == want.shape
        assert np.array_equal(got, want.astype(np.int32)), rank
