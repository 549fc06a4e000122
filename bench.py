"""Benchmark of the W8A8 INT8 linear layer on GB300.

One step = the whole hot path over one batch of synthetic, device-resident
input: per-token INT8 quantization of X (bf16 [M,K]) and the fused int8 GEMM
with the per-token x per-channel dequantization + bias epilogue (bf16 [M,N]).
Weights are quantized per channel once, before timing (post-training, offline).

Default workload: the DiT QKV projection at 768px, batch 1:
M = 2304 image + 256 text tokens = 2560, K = 3072, N = 9216.

Prints ONE JSON line (rank 0).  `value` is INT8 TOPS (2*M*N*K per step over
the device-timed step), `roofline` describes the GEMM kernel against the
measured dense fp16/bf16 tensor peak (the pipe the int8 codes run through on
sm_103a), `cpu_baseline` times the plain C oracle on a bounded row sample on
the host cores, `e2e` repeats the metric through the public API with host
buffers (H2D of X and D2H of Y of every step inside the timed region,
pipelined across consecutive steps on separate streams).

`--impl reference` times the oracle (the reference implementation of this
build) on the host cores instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload qkv768|mlp_up1024|mlp_down1024|tiny|sweep_M<M>_K<K>_N<N>] [--weights int8|w16]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from w8a8_int8_quantized_i8_gb300 import inputs  # noqa: E402

METRIC = "fused W8A8 GEMM INT8 TOPS and % of GB300 dense INT8 peak at DiT shapes"
WORKLOADS = {
    "qkv768": inputs.QKV_768,
    "mlp_up1024": inputs.MLP_UP_1024,
    "mlp_down1024": inputs.MLP_DOWN_1024,
    "tiny": inputs.TINY,
}
# the sweep's shapes as workloads too (sweep_M<M>_K<K>_N<N>), e.g. the
# few-token ones that run the weight-streaming kernel
WORKLOADS.update({sh.name: sh for sh in inputs.sweep_shapes()})
L2_BYTES = 129 * 1024 * 1024
# Dense INT8 rate of this GB300's legacy warp MMA (mma.sync s8 -> s32), the
# chip's INT8 engine, measured by bench_engines.py (profiles/engine_rates.md).
INT8_ENGINE_TOPS = 158.4
# Nominal dense fp8 / bf16 tensor rate on GB300 (4.5 / 2.25 PF/s): the E4M3
# arm's peak is the measured bf16 peak times this ratio.
FP8_OVER_BF16 = 2.0
ROTATE_MIN_BYTES = 3 * L2_BYTES


def _bound(ops, alg_bytes, t_s, tc_peak, hbm_peak):
    """Roofline side of one GEMM launch: "tensor" when its flops at the tensor
    peak take longer than its algorithmic bytes at the HBM peak (the DiT
    shapes), else "hbm" (few tokens: the weights dominate).  Returns
    (bound, achieved, peak, unit)."""
    if ops / (tc_peak * 1e12) >= alg_bytes / (hbm_peak * 1e9):
        return "tensor", ops / t_s / 1e12, tc_peak, "TFLOP/s"
    return "hbm", alg_bytes / t_s / 1e9, hbm_peak, "GB/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# Committed ncu summaries per (arm, workload) and the kernel sources each
# capture was taken from: the DRAM traffic is quoted only while the sources
# still hash to the value recorded in the summary.
PROFILE_SUMMARIES = {
    ("int8", "dit_qkv_768px_M2560_K3072_N9216"): "gemm_w8a8_qkv768_M2560_K3072_N9216.md",
    # few tokens: the int8 arm runs the weight-streaming kernel
    ("int8", "sweep_M1_K3072_N9216"): ("gemm_skinny_M1_K3072_N9216.md", "int8_skinny"),
    ("e4m3", "dit_qkv_768px_M2560_K3072_N9216"): "gemm_direct_e4m3_qkv768_M2560_K3072_N9216.md",
    ("f16codes", "dit_qkv_768px_M2560_K3072_N9216"): "gemm_direct_f16codes_qkv768_M2560_K3072_N9216.md",
}
KERNEL_SOURCES = {
    "int8_skinny": ("w8a8_int8_quantized_i8_gb300/csrc/skinny.cuh",
                    "w8a8_int8_quantized_i8_gb300/csrc/gemm.cuh",
                    "w8a8_int8_quantized_i8_gb300/csrc/ptx.cuh",
                    "w8a8_int8_quantized_i8_gb300/csrc/quant.cuh"),
    "int8": ("w8a8_int8_quantized_i8_gb300/csrc/gemm.cuh",
             "w8a8_int8_quantized_i8_gb300/csrc/gemm_pair.cuh",
             "w8a8_int8_quantized_i8_gb300/csrc/ptx.cuh",
             "w8a8_int8_quantized_i8_gb300/csrc/quant.cuh"),
    "e4m3": ("w8a8_int8_quantized_i8_gb300/csrc/gemm_direct.cuh",
             "w8a8_int8_quantized_i8_gb300/csrc/gemm.cuh",
             "w8a8_int8_quantized_i8_gb300/csrc/ptx.cuh"),
    "f16codes": ("w8a8_int8_quantized_i8_gb300/csrc/gemm_direct.cuh",
                 "w8a8_int8_quantized_i8_gb300/csrc/gemm.cuh",
                 "w8a8_int8_quantized_i8_gb300/csrc/ptx.cuh"),
}


def kernel_sources_sha256(arm: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for src in KERNEL_SOURCES[arm]:
        with open(os.path.join(ROOT, src), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _profiled_traffic(workload: str, arm: str):
    """DRAM bytes per launch of the arm's GEMM from the committed ncu summary,
    or None when no summary covers this workload or the kernel sources
    changed since the capture."""
    name = PROFILE_SUMMARIES.get((arm, workload))
    if name is None:
        return None
    src_arm = arm
    if isinstance(name, tuple):      # (summary, the source set its kernel is built from)
        name, src_arm = name
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and not line.startswith(("|", "#", " ")):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("workload") != workload:
        return None
    if fields.get("kernel_sources_sha256") != kernel_sources_sha256(src_arm):
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return dist, rank, ws, local
    return None, 0, 1, 0


def _max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def _barrier(dist):
    if dist is not None:
        dist.barrier()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if sm:
            out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                   "reasons": sorted(reasons), "samples": len(sm)}
        return out


# --------------------------------------------------------------------- oracle arm
def _oracle_sample(shape, target_s: float):
    """Time the oracle (quant of sampled rows + GEMM against all N weights +
    epilogue) on the host cores; grow the row sample until it takes target_s."""
    import oracle
    oracle.build()
    d = inputs.linear_inputs(shape)
    xb = inputs.bits(d["x"])
    wq, s_w = oracle.quant_rows(inputs.bits(d["w"]))   # offline, like the GPU arm
    bb = inputs.bits(d["bias"])
    rows = 4
    while True:
        t0 = time.perf_counter()
        aq, s_a = oracle.quant_rows(xb[:rows])
        acc = oracle.gemm_s32(aq, wq)
        oracle.dequant_bias(acc, s_a, s_w, bb)
        dt = time.perf_counter() - t0
        if dt >= target_s or rows >= shape.M:
            break
        rows = min(shape.M, max(rows * 2, int(rows * target_s / max(dt, 1e-3) * 0.8)))
    ops = 2.0 * rows * shape.N * shape.K
    return dict(rows=rows, seconds=dt, tops=ops / dt / 1e12, threads=oracle.num_threads(),
                xb=xb, wq=wq, s_w=s_w, bb=bb)


def run_reference(args, shape, dist, rank, world):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    d = inputs.linear_inputs(shape)
    xb = inputs.bits(d["x"])
    wq, s_w = oracle.quant_rows(inputs.bits(d["w"]))
    bb = inputs.bits(d["bias"])
    # rows per step: about 0.25 s of oracle work per step on this host
    rows = 4
    while True:
        t0 = time.perf_counter()
        aq, s_a = oracle.quant_rows(xb[:rows])
        oracle.dequant_bias(oracle.gemm_s32(aq, wq), s_a, s_w, bb)
        dt = time.perf_counter() - t0
        if dt >= 0.2 or rows >= shape.M:
            break
        rows = min(shape.M, rows * 2)
    times = []
    for i in range(args.warmup + args.steps):
        r0 = (i * rows) % max(1, shape.M - rows + 1)
        t0 = time.perf_counter()
        aq, s_a = oracle.quant_rows(xb[r0:r0 + rows])
        oracle.dequant_bias(oracle.gemm_s32(aq, wq), s_a, s_w, bb)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    ops = 2.0 * rows * shape.N * shape.K
    v = ops / t / 1e12
    cores = oracle.num_threads()
    sample = f"{rows} of {shape.M} token rows per step, all N={shape.N} channels, K={shape.K}"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": shape.name, "M": shape.M, "K": shape.K, "N": shape.N},
        "cpu_baseline": {"value": v, "unit": "TOPS", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


# --------------------------------------------------------------------- GPU arm
def run_ours(args, shape, dist, rank, world, local):
    import w8a8_int8_quantized_i8_gb300 as i8
    from w8a8_int8_quantized_i8_gb300 import binding

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = i8.load()
    M, K, N = shape.M, shape.K, shape.N
    hbm_peak, tc_peak, peak_kind = _peaks()

    d = inputs.linear_inputs(shape)
    x_host = d["x"]
    set_bytes = M * K * 2 + M * K + M * 4 + M * N * 2 + N * K * (2 if args.weights == "w16" else 1)
    R = max(2, min(8, -(-ROTATE_MIN_BYTES // set_bytes)))
    sets = []
    w_dev = d["w"].to(dev)
    b_dev = d["bias"].to(dev)
    wq0, s_w = i8.quant_weight_perchannel(w_dev)
    if args.weights == "w16":
        wq0 = i8.widen_weight_codes(wq0)
    ws_bytes = i8.workspace_bytes(M, N, K)
    for r in range(R):
        sets.append(dict(
            x=x_host.to(dev), aq=torch.empty(M, K, dtype=torch.int8, device=dev),
            s_a=torch.empty(M, dtype=torch.float32, device=dev),
            w=wq0.clone(), y=torch.empty(M, N, dtype=torch.bfloat16, device=dev),
            ws=torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)))
    del wq0
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    gemm_fn = lib.i8_gemm_dequant_bias_bf16_w16 if args.weights == "w16" else lib.i8_gemm_dequant_bias_bf16
    vp = ctypes.c_void_p
    calls = []
    for s in sets:
        calls.append((
            (vp(s["x"].data_ptr()), M, K, K, vp(s["aq"].data_ptr()), K, vp(s["s_a"].data_ptr()), sp),
            (vp(s["aq"].data_ptr()), vp(s["s_a"].data_ptr()), vp(s["w"].data_ptr()),
             vp(s_w.data_ptr()), vp(b_dev.data_ptr()), M, N, K, vp(s["y"].data_ptr()), N,
             vp(s["ws"].data_ptr()), ws_bytes, sp)))
    quant_fn = lib.i8_quant_act_pertoken

    def step(i, evq=None, evg=None):
        qa, ga = calls[i % R]
        if evq is not None:
            evq[0].record(stream)
        st = quant_fn(*qa)
        if evg is not None:
            evg[0].record(stream)
        st |= gemm_fn(*ga)
        if evg is not None:
            evg[1].record(stream)
        if st:
            raise RuntimeError(f"libi8 call failed with status {st}")

    for i in range(args.warmup):
        step(i)
    binding.sync_check(dev)

    ev_q = [(torch.cuda.Event(enable_timing=True),) for _ in range(args.steps)]
    ev_g = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    _barrier(dist)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    _barrier(dist)
    # Per-kernel durations: the same K steps again with an event before and
    # after each kernel.  An event between two kernels keeps the second from
    # being scheduled while the first drains, so the headline pass above
    # records none.
    for i in range(args.steps):
        step(i, ev_q[i], ev_g[i])
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    binding.sync_check(dev)
    t_ms = e0.elapsed_time(e1) / args.steps
    t_ms = _max_over_ranks(dist, t_ms)
    gemm_all = sorted(a.elapsed_time(b) for a, b in ev_g)
    gemm_ms = statistics.mean(gemm_all)
    pct = lambda q: gemm_all[min(len(gemm_all) - 1, int(q * len(gemm_all)))] * 1e3
    quant_ms = statistics.mean(q[0].elapsed_time(g[0]) for q, g in zip(ev_q, ev_g))
    ops = 2.0 * M * N * K
    total_ops = _sum_over_ranks(dist, ops * args.steps)
    value = total_ops / (t_ms * 1e-3 * args.steps) / 1e12
    gemm_tops = ops / (gemm_ms * 1e-3) / 1e12
    quant_bytes = 3.0 * M * K + 4.0 * M
    splits = 1 if ws_bytes == 0 else "split-K"
    launches_per_step = 2 + (1 if ws_bytes > 0 else 0)

    # ---- e2e through the public API with host buffers: every step copies
    # its X from pinned host memory and its Y back, pipelined the way a user
    # would run consecutive calls (two buffer sets; copy-in, compute and
    # copy-out on separate streams so step i+1's H2D and step i-1's D2H
    # overlap step i's kernels).
    e2e_steps = max(6, min(args.steps, 60))
    x_pin = [x_host.pin_memory() for _ in range(2)]
    y_pin = [torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    slots = sets[:2]
    s_in = torch.cuda.Stream(dev)
    s_cmp = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def e2e_run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_cmp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            j = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[i - 2])          # X slot free again
                slots[j]["x"].copy_(x_pin[j], non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[i])
                if i >= 2:
                    s_cmp.wait_event(ev_out[i - 2])         # Y slot read back
                i8.linear(slots[j]["x"], slots[j]["w"], s_w, b_dev, out=slots[j]["y"],
                          workspace=slots[j]["ws"] if ws_bytes else None)
                ev_cmp[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[i])
                y_pin[j].copy_(slots[j]["y"], non_blocking=True)
                ev_out[i].record(s_out)
        return ev_out

    e2e_run(4)
    torch.cuda.synchronize(dev)
    _barrier(dist)
    t0 = time.perf_counter()
    evs = e2e_run(e2e_steps)
    evs[-1].synchronize()
    torch.cuda.synchronize(dev)
    e2e_ms = _max_over_ranks(dist, (time.perf_counter() - t0) * 1e3 / e2e_steps)
    e2e_val = _sum_over_ranks(dist, ops) / (e2e_ms * 1e-3) / 1e12

    # ---- the E4M3 (FP8) arm on the same workload: per-token E4M3 quant +
    # the fused E4M3 GEMM, timed the same way (headline pass without events,
    # then a pass with events around each GEMM), rotating the same number of
    # buffer sets.  Reported beside the int8 line, against the FP8 peak.
    e4m3 = None
    if not args.no_e4m3:
        e4m3 = _run_e4m3(args, i8, lib, shape, d, dev, stream, sp, R, tc_peak, peak_kind, local)
    # ---- the same exact W8A8 product with the codes held as fp16 values
    # (quantizer fp16-code output, weights widened offline), no on-chip widening
    f16codes = None
    if not args.no_e4m3:
        f16codes = _run_f16codes(args, i8, lib, shape, d, dev, stream, sp, R, tc_peak, peak_kind, local)

    # ---- oracle on the host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        o = _oracle_sample(shape, target_s=8.0)
        cpu = {"value": o["tops"], "unit": "TOPS", "cores": o["threads"], "kind": "oracle",
               "sample": (f"{o['rows']} of {M} token rows (all N={N} channels, K={K}): "
                          f"quant + int32 GEMM + epilogue in {o['seconds']:.2f} s")}

    # algorithmic bytes of one GEMM launch: codes of A and W, bf16 Y, the
    # scales and the bias
    wbytes = 2 if args.weights == "w16" else 1
    alg_bytes = M * K + wbytes * N * K + 2 * M * N + 4 * M + 6 * N
    rb, ra, rp, ru = _bound(ops, alg_bytes, gemm_ms * 1e-3, tc_peak, hbm_peak)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8", "data": "synthetic",
            "config": {"workload": shape.name, "M": M, "K": K, "N": N,
                       "weights": "int8 codes" if args.weights == "int8" else
                                  "fp16-widened int8 codes (offline)",
                       "l2": f"rotating {R} buffer sets of {set_bytes / 1e6:.0f} MB "
                             f"(inputs of a step last touched {R - 1} steps earlier)",
                       "k_split": splits, "replicas": world},
            "roofline": {"bound": rb, "achieved": ra, "peak": rp, "unit": ru, "frac": ra / rp,
                         "alg_bytes": alg_bytes,
                         "traffic": (_profiled_traffic(shape.name, "int8")
                                     if args.weights == "int8" else None),
                         "traffic_unit": "bytes per launch (ncu dram read + write)",
                         "kernel": "gemm_w8a8 (CTA-pair or single-CTA per the shape table)",
                         "peak_note": f"{peak_kind} dense bf16 burst (same nominal rate as the "
                                      "fp16 kind the int8 codes run through)"},
            "quant_roofline": {"bound": "hbm", "achieved": quant_bytes / (quant_ms * 1e-3) / 1e9,
                               "peak": hbm_peak, "unit": "GB/s",
                               "frac": quant_bytes / (quant_ms * 1e-3) / 1e9 / hbm_peak,
                               "kernel": "quant_rows_kernel", "us": quant_ms * 1e3},
            "gemm_us": gemm_ms * 1e3,
            "gemm_us_p10_p50_p90": [pct(0.1), pct(0.5), pct(0.9)],
            "kernel_timing": "CUDA events around each kernel in a second pass of the same "
                             "steps (the headline pass has no events between kernels)",
            "vs_int8_engine": {"int8_tops_measured": INT8_ENGINE_TOPS, "gemm_ratio": gemm_tops / INT8_ENGINE_TOPS,
                               "source": "mma.sync m16n8k32 s8 rate on this GB300 (bench_engines.py)"},
            "e4m3": e4m3,
            "f16codes": f16codes,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "TOPS", "h2d_bytes_per_step": M * K * 2,
                    "d2h_bytes_per_step": M * N * 2, "ms_per_step": e2e_ms,
                    "how": "public API (i8.linear) with pinned host X/Y, two buffer sets, "
                           "copy-in / compute / copy-out streams, host wall clock"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
        }
        print(json.dumps(line))
    return 0


def _run_e4m3(args, i8, lib, shape, d, dev, stream, sp, R, tc_peak, peak_kind, local):
    """The E4M3 arm: quant + fused GEMM steps on device-resident inputs."""
    from w8a8_int8_quantized_i8_gb300 import binding
    M, K, N = shape.M, shape.K, shape.N
    vp = ctypes.c_void_p
    wq, s_w = i8.quant_weight_perchannel_e4m3(d["w"].to(dev))
    wq = wq.view(torch.uint8)
    b_dev = d["bias"].to(dev)
    ws_bytes = i8.e4m3_workspace_bytes(M, N, K)
    sets = [dict(x=d["x"].to(dev), aq=torch.empty(M, K, dtype=torch.uint8, device=dev),
                 s_a=torch.empty(M, dtype=torch.float32, device=dev),
                 w=wq.clone(), y=torch.empty(M, N, dtype=torch.bfloat16, device=dev),
                 ws=torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev))
            for _ in range(R)]
    calls = [((vp(t["x"].data_ptr()), M, K, K, vp(t["aq"].data_ptr()), K, vp(t["s_a"].data_ptr()), sp),
              (vp(t["aq"].data_ptr()), vp(t["s_a"].data_ptr()), vp(t["w"].data_ptr()),
               vp(s_w.data_ptr()), vp(b_dev.data_ptr()), M, N, K, vp(t["y"].data_ptr()), N,
               vp(t["ws"].data_ptr()), ws_bytes, sp))
             for t in sets]
    qf, gf = lib.i8_quant_act_pertoken_e4m3, lib.i8_gemm_e4m3_dequant_bias_bf16

    def step(i, evg=None):
        qa, ga = calls[i % R]
        st = qf(*qa)
        if evg is not None:
            evg[0].record(stream)
        st |= gf(*ga)
        if evg is not None:
            evg[1].record(stream)
        if st:
            raise RuntimeError(f"libi8 E4M3 call failed with status {st}")

    steps = max(10, min(args.steps, 1000))
    for i in range(max(3, args.warmup)):
        step(i)
    binding.sync_check(dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    evg = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        step(i, evg[i])
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    binding.sync_check(dev)
    ops = 2.0 * M * N * K
    t_ms = e0.elapsed_time(e1) / steps
    g_ms = statistics.mean(a.elapsed_time(b) for a, b in evg)
    peak = tc_peak * FP8_OVER_BF16
    g_tflops = ops / (g_ms * 1e-3) / 1e12
    alg_bytes = M * K + N * K + 2 * M * N + 4 * M + 6 * N
    rb, ra, rp, ru = _bound(ops, alg_bytes, g_ms * 1e-3, peak, _peaks()[0])
    return {
        "value": ops / (t_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": t_ms, "steps": steps,
        "dtype": "e4m3", "gemm_us": g_ms * 1e3,
        "roofline": {"bound": rb, "achieved": ra, "peak": rp, "unit": ru, "frac": ra / rp,
                     "alg_bytes": alg_bytes, "traffic": _profiled_traffic(shape.name, "e4m3"),
                     "traffic_unit": "bytes per launch (ncu dram read + write)",
                     "kernel": "gemm_direct_pair_kernel<E4M3>",
                     "peak_note": f"{peak_kind} dense bf16 burst x {FP8_OVER_BF16:g} "
                                  "(nominal dense fp8 / bf16 rate: 4.5 / 2.25 PF/s)"},
        "parity": "codes bit-exact; fp32 accumulators within the derived rounding bound of the "
                  "exact sum; bf16 = oracle epilogue of the GPU accumulators, bit for bit",
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
    }


def _run_f16codes(args, i8, lib, shape, d, dev, stream, sp, R, tc_peak, peak_kind, local):
    """The exact path with fp16-held codes: quant (fp16 codes) + fused GEMM."""
    from w8a8_int8_quantized_i8_gb300 import binding
    M, K, N = shape.M, shape.K, shape.N
    vp = ctypes.c_void_p
    wq, s_w = i8.quant_weight_perchannel(d["w"].to(dev))
    w16 = i8.widen_weight_codes(wq)
    del wq
    b_dev = d["bias"].to(dev)
    ws_bytes = i8.f16codes_workspace_bytes(M, N, K)
    sets = [dict(x=d["x"].to(dev), aq=torch.empty(M, K, dtype=torch.float16, device=dev),
                 s_a=torch.empty(M, dtype=torch.float32, device=dev),
                 w=w16.clone(), y=torch.empty(M, N, dtype=torch.bfloat16, device=dev),
                 ws=torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev))
            for _ in range(R)]
    del w16
    calls = [((vp(t["x"].data_ptr()), M, K, K, vp(t["aq"].data_ptr()), K, vp(t["s_a"].data_ptr()), sp),
              (vp(t["aq"].data_ptr()), vp(t["s_a"].data_ptr()), vp(t["w"].data_ptr()),
               vp(s_w.data_ptr()), vp(b_dev.data_ptr()), M, N, K, vp(t["y"].data_ptr()), N,
               vp(t["ws"].data_ptr()), ws_bytes, sp))
             for t in sets]
    qf, gf = lib.i8_quant_act_pertoken_f16codes, lib.i8_gemm_dequant_bias_bf16_f16codes

    def step(i, evg=None):
        qa, ga = calls[i % R]
        st = qf(*qa)
        if evg is not None:
            evg[0].record(stream)
        st |= gf(*ga)
        if evg is not None:
            evg[1].record(stream)
        if st:
            raise RuntimeError(f"libi8 fp16-code call failed with status {st}")

    steps = max(10, min(args.steps, 1000))
    for i in range(max(3, args.warmup)):
        step(i)
    binding.sync_check(dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    evg = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        step(i, evg[i])
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    binding.sync_check(dev)
    ops = 2.0 * M * N * K
    t_ms = e0.elapsed_time(e1) / steps
    g_ms = statistics.mean(a.elapsed_time(b) for a, b in evg)
    g_tops = ops / (g_ms * 1e-3) / 1e12
    alg_bytes = 2 * M * K + 2 * N * K + 2 * M * N + 4 * M + 6 * N
    rb, ra, rp, ru = _bound(ops, alg_bytes, g_ms * 1e-3, tc_peak, _peaks()[0])
    return {
        "value": ops / (t_ms * 1e-3) / 1e12, "unit": "TOPS", "ms_per_step": t_ms, "steps": steps,
        "dtype": "int8 codes held as fp16 (exact int32 accumulation)", "gemm_us": g_ms * 1e3,
        "bytes_note": "activation codes 2 B (written by the quantizer), weight codes 2 B (widened offline)",
        "roofline": {"bound": rb, "achieved": ra, "peak": rp, "unit": ru, "frac": ra / rp,
                     "alg_bytes": alg_bytes, "traffic": _profiled_traffic(shape.name, "f16codes"),
                     "traffic_unit": "bytes per launch (ncu dram read + write)",
                     "kernel": "gemm_direct_pair_kernel<F16 codes>",
                     "peak_note": f"{peak_kind} dense bf16 burst (the fp16 kind's nominal rate)"},
        "parity": "int32 and bf16 bit-identical to the oracle and to the int8-code kernels",
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="qkv768")
    ap.add_argument("--weights", choices=["int8", "w16"], default="int8")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-e4m3", action="store_true",
                    help="skip the E4M3 (FP8) arm and the fp16-code variant")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    shape = WORKLOADS[args.workload]
    dist, rank, world, local = _dist()
    try:
        if args.impl == "reference":
            return run_reference(args, shape, dist, rank, world)
        return run_ours(args, shape, dist, rank, world, local)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
