"""The bench's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

The path shards without any exchange (replicas), so the only multi-rank
logic is the barrier around the timed region, the max-over-ranks step time,
the sum-over-ranks work, and the rule that the reference arm runs on rank 0
only.  No GPU is involved.
"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    dist, r, w, local = bench._dist()
    assert (r, w, local) == (rank, world, rank)
    bench._barrier(dist)
    t_max = bench._max_over_ranks(dist, 1.0 + rank)        # rank 1 is the slow one
    work = bench._sum_over_ranks(dist, 100.0 * (rank + 1))
    # value = all ranks' work / the slowest rank's time
    q.put((rank, t_max, work, work / t_max))
    dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, work, value in out:
        assert t_max == 2.0          # max over ranks, not the local time
        assert work == 300.0         # sum over ranks
        assert value == 150.0


def _ref_worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import contextlib
    import io
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    q.put((rank, rc, buf.getvalue()))


def test_reference_arm_runs_on_rank_zero_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ref_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, rc0, s0), (r1, rc1, s1) = out
    assert rc0 == 0 and rc1 == 0
    assert '"impl": "reference"' in s0 and s0.count("\n") == 1
    assert s1 == ""


def test_roofline_side_follows_arithmetic_intensity():
    """The bench reports a GEMM against the tensor peak when its flops at that
    peak outlast its bytes at the HBM peak, else against HBM bandwidth."""
    import bench
    tc, hbm = 1924.1, 6794.5
    # DiT QKV at 768px: 145 GOP, 83 MB -> tensor side
    side, achieved, peak, unit = bench._bound(2 * 2560 * 9216 * 3072, 83.4e6, 112.6e-6, tc, hbm)
    assert (side, unit, peak) == ("tensor", "TFLOP/s", tc)
    assert abs(achieved - 2 * 2560 * 9216 * 3072 / 112.6e-6 / 1e12) < 1e-6
    # one token against the same weights: 57 MOP, 28 MB -> HBM side
    side, achieved, peak, unit = bench._bound(2 * 1 * 9216 * 3072, 28.4e6, 13e-6, tc, hbm)
    assert (side, unit, peak) == ("hbm", "GB/s", hbm)
    assert abs(achieved - 28.4e6 / 13e-6 / 1e9) < 1e-6


def test_profile_lookup_uses_the_summarys_source_set(tmp_path, monkeypatch):
    """A capture's DRAM traffic (profiles/traffic.json) is quoted only while
    the kernel sources of its source set still hash to the recorded value."""
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for src in set(bench.KERNEL_SOURCES["int8_skinny"]):
        p = tmp_path / src
        p.parent.mkdir(parents=True, exist_ok=True)
        p.write_text("// " + src)
    import json
    sha = bench.kernel_sources_sha256("int8_skinny")
    (prof / "traffic.json").write_text(json.dumps({"entries": [
        {"arm": "int8", "workload": "sweep_M1_K3072_N9216", "source_set": "int8_skinny",
         "traffic_bytes_per_launch": 123, "kernel_sources_sha256": sha}]}))
    assert bench._profiled_traffic("sweep_M1_K3072_N9216", "int8") == 123
    (tmp_path / bench.KERNEL_SOURCES["int8_skinny"][0]).write_text("// changed")
    assert bench._profiled_traffic("sweep_M1_K3072_N9216", "int8") is None
    assert bench._profiled_traffic("no_such_workload", "int8") is None


def test_reference_arm_line_keeps_the_contract(capsys, monkeypatch):
    """One process: the reference arm's JSON line carries every key of the
    bench contract, with the oracle's own figures in cpu_baseline and e2e."""
    import json
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"])
    assert rc == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2
    assert d["warmup"] >= 3                      # raised to the contract's minimum
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    assert "workload" in d["config"]
    cb, e2e = d["cpu_baseline"], d["e2e"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert e2e == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}
