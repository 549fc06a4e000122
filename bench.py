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

Beside the headline the line carries, from the same process:
* ``configs``: the DiT MLP pair at 1024px, batch 2 (up 8704 x 3072 x 12288,
  down 8704 x 12288 x 3072 on GELU inputs) timed the same way, each with its
  GEMM and quantizer rooflines; one few-token shape (1 x 3072 x 9216, the
  weight-streaming kernel) against HBM; and the synthetic 28-block DiT linear
  stack at 1024px, batch 2 (linear-layer time per denoising step);
* ``library``: torch bf16 ``addmm`` (cuBLAS), ``torch._int_mm`` and the
  "fake INT8" forward (both operands dequantized to bf16, then a bf16 matmul)
  on the same inputs, at the headline workload and at the MLP pair;
* ``int8_engine``: the rate of this GPU's int8 tensor instruction (the legacy
  warp MMA, mma.sync s8), measured in this run;
* ``cosine``: the headline output against the fake-INT8 forward and against
  the unquantized bf16 product, with NaN/Inf counts.

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


# DRAM traffic per launch of each arm's GEMM from the committed ncu captures
# (profiles/traffic.json), quoted only while the kernel sources still hash to
# the value recorded with the capture.
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
TRAFFIC_NOTE = ("ncu dram read + write bytes of one captured launch; ncu flushes the caches "
                "before the launch, so output still held in L2 when the kernel ends is not counted")


def kernel_sources_sha256(arm: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for src in KERNEL_SOURCES[arm]:
        with open(os.path.join(ROOT, src), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _profiled_traffic(workload: str, arm: str):
    """DRAM bytes per launch of the arm's GEMM on this workload from the
    committed captures, or None when none covers it or the kernel sources
    changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            entries = json.load(fh)["entries"]
    except (OSError, ValueError, KeyError):
        return None
    for e in entries:
        if e.get("arm") == arm and e.get("workload") == workload:
            if e.get("kernel_sources_sha256") != kernel_sources_sha256(e.get("source_set", arm)):
                return None
            return int(e["traffic_bytes_per_launch"])
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
def _setup_int8(i8, lib, shape, d, dev, stream, weights="int8"):
    """Device buffers for the int8 path on one workload: weights quantized
    once (offline), and enough rotating sets of (X, A_q, s_a, W_q, Y,
    workspace) that a step's inputs were last touched more than 3 x L2 of
    traffic earlier.  Returns the context the timers use."""
    M, K, N = shape.M, shape.K, shape.N
    set_bytes = M * K * 2 + M * K + M * 4 + M * N * 2 + N * K * (2 if weights == "w16" else 1)
    R = max(2, min(8, -(-ROTATE_MIN_BYTES // set_bytes)))
    w_dev = d["w"].to(dev)
    b_dev = d["bias"].to(dev)
    wq0, s_w = i8.quant_weight_perchannel(w_dev)
    del w_dev
    if weights == "w16":
        wq0 = i8.widen_weight_codes(wq0)
    ws_bytes = i8.workspace_bytes(M, N, K)
    x_dev = d["x"].to(dev)
    sets = []
    for r in range(R):
        sets.append(dict(
            x=x_dev if r == 0 else x_dev.clone(),
            aq=torch.empty(M, K, dtype=torch.int8, device=dev),
            s_a=torch.empty(M, dtype=torch.float32, device=dev),
            w=wq0 if r == 0 else wq0.clone(), y=torch.empty(M, N, dtype=torch.bfloat16, device=dev),
            ws=torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)))
    sp = ctypes.c_void_p(stream.cuda_stream)
    vp = ctypes.c_void_p
    calls = []
    for t in sets:
        calls.append((
            (vp(t["x"].data_ptr()), M, K, K, vp(t["aq"].data_ptr()), K, vp(t["s_a"].data_ptr()), sp),
            (vp(t["aq"].data_ptr()), vp(t["s_a"].data_ptr()), vp(t["w"].data_ptr()),
             vp(s_w.data_ptr()), vp(b_dev.data_ptr()), M, N, K, vp(t["y"].data_ptr()), N,
             vp(t["ws"].data_ptr()), ws_bytes, sp)))
    gemm_fn = lib.i8_gemm_dequant_bias_bf16_w16 if weights == "w16" else lib.i8_gemm_dequant_bias_bf16
    return dict(shape=shape, sets=sets, calls=calls, R=R, set_bytes=set_bytes, ws_bytes=ws_bytes,
                s_w=s_w, b_dev=b_dev, weights=weights, quant_fn=lib.i8_quant_act_pertoken,
                gemm_fn=gemm_fn)


def _time_int8(ctx, stream, dev, steps, warmup, dist=None):
    """Time `steps` steps (per-token quant + fused GEMM) back to back with no
    event between kernels, then the same steps again with events around each
    kernel, then each kernel alone back to back."""
    calls, R = ctx["calls"], ctx["R"]
    qf, gf = ctx["quant_fn"], ctx["gemm_fn"]

    def step(i, evq=None, evg=None):
        qa, ga = calls[i % R]
        if evq is not None:
            evq.record(stream)
        st = qf(*qa)
        if evg is not None:
            evg[0].record(stream)
        st |= gf(*ga)
        if evg is not None:
            evg[1].record(stream)
        if st:
            raise RuntimeError(f"libi8 call failed with status {st}")

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    ev_q = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev_g = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(steps)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    _barrier(dist)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    _barrier(dist)
    # Per-kernel durations: the same steps again with an event before and
    # after each kernel.  An event between two kernels keeps the second from
    # being scheduled while the first drains, so the headline pass records none.
    for i in range(steps):
        step(i, ev_q[i], ev_g[i])
    torch.cuda.synchronize(dev)
    # Each kernel alone, `steps` launches back to back over the rotating sets
    # with events only at the ends of the pass: its average launch duration
    # when launches follow one another, as in a chain of layers.  (An event
    # right before a launch adds the launch latency that a launch queued
    # behind another kernel hides: 4-5 us on this GPU for an empty kernel.)
    pass_ms = []
    for which in (0, 1):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            st = (qf if which == 0 else gf)(*calls[i % R][which])
            if st:
                raise RuntimeError(f"libi8 call failed with status {st}")
        b.record(stream)
        torch.cuda.synchronize(dev)
        pass_ms.append(a.elapsed_time(b) / steps)
    t_ms = e0.elapsed_time(e1) / steps
    gemm_all = sorted(a.elapsed_time(b) for a, b in ev_g)
    quant_ms = statistics.mean(q.elapsed_time(g[0]) for q, g in zip(ev_q, ev_g))
    return dict(step_ms=t_ms, gemm_bracketed=gemm_all, quant_bracketed_ms=quant_ms,
                quant_ms=pass_ms[0], gemm_ms=pass_ms[1])


def _gemm_roofline(shape, gemm_ms, tc_peak, hbm_peak, peak_kind, wbytes=1, arm="int8"):
    M, K, N = shape.M, shape.K, shape.N
    ops = 2.0 * M * N * K
    # algorithmic bytes of one GEMM launch: codes of A and W, bf16 Y, the
    # scales and the bias
    alg_bytes = M * K + wbytes * N * K + 2 * M * N + 4 * M + 6 * N
    rb, ra, rp, ru = _bound(ops, alg_bytes, gemm_ms * 1e-3, tc_peak, hbm_peak)
    return {"bound": rb, "achieved": ra, "peak": rp, "unit": ru, "frac": ra / rp,
            "alg_bytes": alg_bytes,
            "traffic": _profiled_traffic(shape.name, arm) if wbytes == 1 else None,
            "traffic_unit": "bytes per launch", "traffic_note": TRAFFIC_NOTE,
            "kernel": "gemm_w8a8 (CTA-pair, single-CTA or few-token kernel per the shape table)",
            "peak_note": (f"{peak_kind} dense bf16 burst (same nominal rate as the fp16 kind the "
                          "int8 codes run through)" if rb == "tensor" else f"{peak_kind} HBM copy")}


def _quant_roofline(shape, tm, hbm_peak):
    qb = 3.0 * shape.M * shape.K + 4.0 * shape.M
    gbs = qb / (tm["quant_ms"] * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
            "alg_bytes": qb, "kernel": "quant_rows_kernel", "us": tm["quant_ms"] * 1e3,
            "us_event_bracketed": tm["quant_bracketed_ms"] * 1e3,
            "timing": "average launch duration over a pass of back-to-back quantizer launches "
                      "(rotating L2-cold inputs); us_event_bracketed: mean of single launches "
                      "with an event right before and after each"}


def _gemm_fields(tm):
    g = tm["gemm_bracketed"]
    return {"gemm_us": tm["gemm_ms"] * 1e3,
            "gemm_us_event_bracketed": statistics.mean(g) * 1e3,
            "gemm_us_event_bracketed_p10_p50_p90": [g[int(q * (len(g) - 1))] * 1e3 for q in (0.1, 0.5, 0.9)]}


def _pass_ms(fn, n, stream):
    """Average device time of fn(i) over n calls back to back, events only at
    the ends of the pass (the way the library's kernels are timed)."""
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(n):
        fn(i)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def _library_comparisons(ctx, d, stream, n, gemm_ms):
    """torch bf16 addmm (cuBLAS), torch._int_mm and the pages' fake-INT8
    forward on the same rotating inputs, each timed like the library's GEMM
    (a pass of back-to-back calls, events at its ends)."""
    shape = ctx["shape"]
    M, K, N = shape.M, shape.K, shape.N
    ops = 2.0 * M * N * K
    R, sets = ctx["R"], ctx["sets"]
    b, s_w = ctx["b_dev"], ctx["s_w"]
    w_bf16 = d["w"].to(stream.device)
    wts = [w_bf16.t()] + [w_bf16.clone().t() for _ in range(R - 1)]
    ys = [torch.empty(M, N, dtype=torch.bfloat16, device=stream.device) for _ in range(R)]
    out = {}
    t = _pass_ms(lambda i: torch.addmm(b, sets[i % R]["x"], wts[i % R], out=ys[i % R]), n, stream)
    out["torch_bf16_addmm"] = {"us": t * 1e3, "tflops": ops / (t * 1e-3) / 1e12,
                               "int8_gemm_speedup": t / gemm_ms}
    if M > 16:
        wqt = [s_["w"].t() for s_ in sets]
        t = _pass_ms(lambda i: torch._int_mm(sets[i % R]["aq"], wqt[i % R]), n, stream)
        out["torch_int_mm"] = {"us": t * 1e3, "tops": ops / (t * 1e-3) / 1e12,
                               "int8_gemm_speedup": t / gemm_ms, "output": "int32 only, no epilogue"}
    s_w16 = s_w.to(torch.bfloat16)[:, None]

    def fake(i):
        r = sets[i % R]
        a_deq = r["aq"].to(torch.bfloat16) * r["s_a"].to(torch.bfloat16)[:, None]
        w_deq = r["w"].to(torch.bfloat16) * s_w16
        torch.addmm(b, a_deq, w_deq.t(), out=ys[i % R])

    t = _pass_ms(fake, n, stream)
    out["fake_int8"] = {"us": t * 1e3, "tops": ops / (t * 1e-3) / 1e12, "int8_gemm_speedup": t / gemm_ms,
                        "what": "dequantize A_q and W_q to bf16, then bf16 addmm (torch ops)"}
    out["timing"] = ("a pass of back-to-back calls over the library's rotating inputs, events at "
                     "its ends; int8_gemm_speedup = that time / the library GEMM's gemm_us")
    del wts, ys
    return out


def _cosines(ctx, d, i8):
    """The pages report cosine 1.0 and no NaN against the reference: the
    library's output against the fake-INT8 forward and against the
    unquantized bf16 product, on the headline inputs (informational)."""
    t = ctx["sets"][0]
    y = i8.linear(t["x"], t["w"], ctx["s_w"], ctx["b_dev"]).double()
    w_bf16 = d["w"].to(t["x"].device)
    b = ctx["b_dev"]
    aq, s_a = i8.quant_act_pertoken(t["x"])
    fake = torch.addmm(b, (aq.to(torch.bfloat16) * s_a.to(torch.bfloat16)[:, None]),
                       (t["w"].to(torch.bfloat16) * ctx["s_w"].to(torch.bfloat16)[:, None]).t()).double()
    ref = torch.addmm(b, t["x"], w_bf16.t()).double()

    def cos(a, c):
        return float((a * c).sum() / (a.norm() * c.norm()))

    return {"vs_fake_int8": cos(y, fake), "vs_bf16_unquantized": cos(y, ref),
            "nan_or_inf": int((~torch.isfinite(y)).sum().item()),
            "what": "cosine of the fused W8A8 output (fp64) with each reference, all M x N elements"}


def _int8_engine(stream):
    """Rate of the int8 tensor instruction of this GPU (mma.sync m16n8k32
    s8 -> s32, register-only loop), measured now."""
    from w8a8_int8_quantized_i8_gb300 import build as _b
    try:
        lib = ctypes.CDLL(_b.PROBE_LIB)
    except OSError as e:
        return {"error": f"libi8probe.so not loaded: {e}"}
    sink = torch.zeros(1, dtype=torch.int32, device=stream.device)
    s8 = ctypes.c_double(0.0)
    f16 = ctypes.c_double(0.0)
    lib.i8probe_mma_rates.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                      ctypes.c_void_p]
    rc = lib.i8probe_mma_rates(3, 256, ctypes.c_void_p(sink.data_ptr()), ctypes.byref(s8),
                               ctypes.byref(f16), ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        return {"error": f"probe returned {rc}"}
    return {"mma_sync_s8_tops": s8.value, "mma_sync_f16_tflops": f16.value,
            "how": "register-only loops of mma.sync m16n8k32 s8 (and m16n8k16 f16), 4 CTAs of "
                   "256 threads per SM, best of 3 launches, measured in this run"}


def _stack_config(i8, dev, steps):
    """Linear-layer time per denoising step of the synthetic 28-block DiT
    stack at 1024px, batch 2 (M = 8704): the sum over its 112 layers of each
    layer's per-token quantizer + fused GEMM, timed with events around each
    layer; the LayerNorm / GELU / V-slice glue runs in torch between the
    timed layers and is excluded."""
    from w8a8_int8_quantized_i8_gb300 import dit_stack
    M = 8704
    stack = dit_stack.build(blocks=28, seed=5, device=dev)
    h = inputs.activations(M, dit_stack.WIDTH, torch.Generator().manual_seed(5)).to(dev)
    events = []

    def timer(begin):
        ev = torch.cuda.Event(enable_timing=True)
        ev.record()
        events.append(ev)

    dit_stack.forward(stack, h)   # warm-up
    torch.cuda.synchronize(dev)
    lin, tot = [], []
    for _ in range(steps):
        events.clear()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        dit_stack.forward(stack, h, timer=timer)
        e1.record()
        torch.cuda.synchronize(dev)
        lin.append(sum(events[i].elapsed_time(events[i + 1]) for i in range(0, len(events), 2)))
        tot.append(e0.elapsed_time(e1))
    i8.sync_check(dev)
    ops = 2.0 * M * 28 * sum(K * N for _, K, N in dit_stack.LAYERS)
    lin_ms = statistics.median(lin)
    del stack
    torch.cuda.empty_cache()
    return {"workload": "dit_linear_stack_1024px_b2_28blocks_M8704", "layers": 112,
            "linear_ms_per_step": lin_ms, "linear_tops": ops / (lin_ms * 1e-3) / 1e12,
            "step_ms_with_glue": statistics.median(tot), "steps": steps,
            "how": "sum of the 112 layers' quant + GEMM times (events around each layer), median "
                   "over steps; torch LayerNorm / GELU / V-slice glue excluded"}


def _config_entry(i8, lib, shape, dev, stream, steps, warmup, tc_peak, hbm_peak, peak_kind, library):
    d = inputs.linear_inputs(shape)
    ctx = _setup_int8(i8, lib, shape, d, dev, stream)
    tm = _time_int8(ctx, stream, dev, steps, warmup)
    t_ms, gemm_ms = tm["step_ms"], tm["gemm_ms"]
    ops = 2.0 * shape.M * shape.N * shape.K
    e = {"M": shape.M, "K": shape.K, "N": shape.N, "value": ops / (t_ms * 1e-3) / 1e12, "unit": "TOPS",
         "ms_per_step": t_ms, **_gemm_fields(tm),
         "roofline": _gemm_roofline(shape, gemm_ms, tc_peak, hbm_peak, peak_kind),
         "quant_roofline": _quant_roofline(shape, tm, hbm_peak),
         "plan": i8.plan_query(shape.M, shape.N, shape.K, "int8")["kernel"],
         "l2": f"rotating {ctx['R']} buffer sets of {ctx['set_bytes'] / 1e6:.0f} MB"}
    if library:
        e["library"] = _library_comparisons(ctx, d, stream, max(10, min(steps, 50)), gemm_ms)
    i8.sync_check(dev)
    del ctx
    torch.cuda.empty_cache()
    return e


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
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    ctx = _setup_int8(i8, lib, shape, d, dev, stream, args.weights)
    R, ws_bytes, set_bytes = ctx["R"], ctx["ws_bytes"], ctx["set_bytes"]
    sets, s_w, b_dev = ctx["sets"], ctx["s_w"], ctx["b_dev"]
    binding.sync_check(dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    tm = _time_int8(ctx, stream, dev, args.steps, args.warmup, dist)
    clk = clocks.stop()
    binding.sync_check(dev)
    t_ms = _max_over_ranks(dist, tm["step_ms"])
    gemm_ms = tm["gemm_ms"]
    ops = 2.0 * M * N * K
    total_ops = _sum_over_ranks(dist, ops * args.steps)
    value = total_ops / (t_ms * 1e-3 * args.steps) / 1e12
    gemm_tops = ops / (gemm_ms * 1e-3) / 1e12
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

    extras = {}
    if rank == 0 and not args.no_extras:
        # ---- same-run comparisons on the headline workload: library GEMMs,
        # the pages' cosine, the int8 tensor instruction's rate
        extras["library"] = _library_comparisons(ctx, d, stream, max(10, min(args.steps, 50)), gemm_ms)
        extras["cosine"] = _cosines(ctx, d, i8)
        extras["int8_engine"] = _int8_engine(stream)
    del ctx, sets, slots
    torch.cuda.empty_cache()

    # ---- the E4M3 (FP8) arm and the exact path with fp16-held codes on the
    # same workload, timed the same way, reported beside the int8 line
    e4m3 = f16codes = None
    if not args.no_e4m3:
        e4m3 = _run_e4m3(args, i8, lib, shape, d, dev, stream, sp, R, tc_peak, peak_kind, local)
        f16codes = _run_f16codes(args, i8, lib, shape, d, dev, stream, sp, R, tc_peak, peak_kind, local)

    # ---- the other DiT configurations (rank 0): MLP pair at 1024px, one
    # few-token shape, the 28-block stack
    configs = None
    if rank == 0 and not args.no_extras:
        configs = {}
        cclk = ClockSampler(local)
        cclk.start()
        for cs, lib_cmp in ((inputs.MLP_UP_1024, True), (inputs.MLP_DOWN_1024, True),
                            (WORKLOADS["sweep_M1_K3072_N9216"], False)):
            configs[cs.name] = _config_entry(i8, lib, cs, dev, stream, args.steps, args.warmup,
                                             tc_peak, hbm_peak, peak_kind, lib_cmp)
        st = _stack_config(i8, dev, max(3, min(args.steps, 5)))
        configs[st.pop("workload")] = st
        c = cclk.stop()
        configs["clocks"] = {k: c[k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")}

    # ---- oracle on the host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        o = _oracle_sample(shape, target_s=8.0)
        cpu = {"value": o["tops"], "unit": "TOPS", "cores": o["threads"], "kind": "oracle",
               "sample": (f"{o['rows']} of {M} token rows (all N={N} channels, K={K}): "
                          f"quant + int32 GEMM + epilogue in {o['seconds']:.2f} s")}

    wbytes = 2 if args.weights == "w16" else 1
    if rank == 0:
        eng = extras.get("int8_engine", {}).get("mma_sync_s8_tops")
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
            "roofline": _gemm_roofline(shape, gemm_ms, tc_peak, hbm_peak, peak_kind, wbytes),
            "quant_roofline": _quant_roofline(shape, tm, hbm_peak),
            **_gemm_fields(tm),
            "kernel_timing": ("value / ms_per_step: K steps (quant + GEMM) back to back, events "
                              "only at the ends.  gemm_us (the roofline's time) and the quantizer's "
                              "us: each kernel alone, K launches back to back over the same "
                              "rotating sets, events only at the ends of the pass (average launch "
                              "duration).  *_event_bracketed: a pass with an event right before "
                              "and after every launch, which adds the launch latency that a "
                              "launch queued behind other work hides"),
            "int8_engine": extras.get("int8_engine"),
            "vs_int8_engine": ({"gemm_ratio": gemm_tops / eng, "int8_tops_measured": eng}
                               if eng else None),
            "library": extras.get("library"),
            "cosine": extras.get("cosine"),
            "e4m3": e4m3,
            "f16codes": f16codes,
            "configs": configs,
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
    # the GEMM alone, back to back over the rotating sets (average launch duration)
    g_ms = _pass_ms(lambda i: gf(*calls[i % R][1]), steps, stream)
    clk = clocks.stop()
    binding.sync_check(dev)
    ops = 2.0 * M * N * K
    t_ms = e0.elapsed_time(e1) / steps
    g_br = statistics.mean(a.elapsed_time(b) for a, b in evg)
    peak = tc_peak * FP8_OVER_BF16
    g_tflops = ops / (g_ms * 1e-3) / 1e12
    alg_bytes = M * K + N * K + 2 * M * N + 4 * M + 6 * N
    rb, ra, rp, ru = _bound(ops, alg_bytes, g_ms * 1e-3, peak, _peaks()[0])
    return {
        "value": ops / (t_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": t_ms, "steps": steps,
        "dtype": "e4m3", "gemm_us": g_ms * 1e3, "gemm_us_event_bracketed": g_br * 1e3,
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
    # the GEMM alone, back to back over the rotating sets (average launch duration)
    g_ms = _pass_ms(lambda i: gf(*calls[i % R][1]), steps, stream)
    clk = clocks.stop()
    binding.sync_check(dev)
    ops = 2.0 * M * N * K
    t_ms = e0.elapsed_time(e1) / steps
    g_br = statistics.mean(a.elapsed_time(b) for a, b in evg)
    g_tops = ops / (g_ms * 1e-3) / 1e12
    alg_bytes = 2 * M * K + 2 * N * K + 2 * M * N + 4 * M + 6 * N
    rb, ra, rp, ru = _bound(ops, alg_bytes, g_ms * 1e-3, tc_peak, _peaks()[0])
    return {
        "value": ops / (t_ms * 1e-3) / 1e12, "unit": "TOPS", "ms_per_step": t_ms, "steps": steps,
        "dtype": "int8 codes held as fp16 (exact int32 accumulation)", "gemm_us": g_ms * 1e3,
        "gemm_us_event_bracketed": g_br * 1e3,
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
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other DiT configurations, the library comparisons, the "
                         "cosines and the int8 engine rate")
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
