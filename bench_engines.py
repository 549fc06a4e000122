"""Comparison measurements on the same GB300: engine rates and the DiT shapes.

Prints one JSON object per line:

* ``engine``: peak rates of the legacy warp MMA on this chip (register-only
  loops of mma.sync m16n8k32 s8->s32 and m16n8k16 f16->f32), compiled here
  from the CUDA source below with nvcc;
* ``shape``: for each DiT linear shape, the device time (calls captured in a
  CUDA graph and replayed) of
  - this library's full step (per-token quant + fused GEMM) and GEMM alone,
    with int8 weights and with pre-widened (fp16-code) weights,
  - torch bf16 ``X @ W.T + b`` (cuBLAS),
  - ``torch._int_mm`` (int32 only, the pages' exactness reference),
  - the "fake INT8" forward the pages replace: dequantize A_q and W_q to bf16,
    then a bf16 matmul + bias (all torch ops);
  inputs rotate over enough buffer sets to exceed 3x the 129 MB L2;
* ``stack`` (with --stack): the linear-layer time per denoising step of the
  synthetic 28-block DiT stack at 1024px batch 2 (M = 8704), int8 and E4M3
  codes, with torch LN/GELU glue and with the fused producer-quantizers.

Usage: python bench_engines.py [--sweep] [--stack] [--no-engines] [--iters N]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import w8a8_int8_quantized_i8_gb300 as i8  # noqa: E402
from w8a8_int8_quantized_i8_gb300 import inputs  # noqa: E402

MMA_SYNC_SRC = r"""
#include <cstdio>
#include <cuda_runtime.h>
__global__ void mma_s8(int iters, int* out) {
  int a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 ^ 5, a3 = a0 + 7, b0 = a0 * 11, b1 = a0 - 1;
  int c[4][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                   : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                   : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
  for (int j = 0; j < 4; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  if (s == 123456789) out[0] = s;
}
__global__ void mma_f16(int iters, int* out) {
  unsigned a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 ^ 5, a3 = a0 + 7, b0 = a0 * 11, b1 = a0 - 1;
  float c[4][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                   : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
                   : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  float s = 0;
  for (int j = 0; j < 4; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  if (s == 123456789.f) out[0] = 1;
}
int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  int* out;
  cudaMalloc(&out, 4);
  const int iters = 4096, blocks = sms * 4, threads = 256;
  double best_s8 = 0, best_f16 = 0;
  for (int rep = 0; rep < 3; ++rep) {
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    float ms;
    const double warps = blocks * threads / 32.0;
    cudaEventRecord(e0);
    mma_s8<<<blocks, threads>>>(iters, out);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    cudaEventElapsedTime(&ms, e0, e1);
    double v = 2.0 * 16 * 8 * 32 * 4.0 * iters * warps / ms / 1e9;
    if (v > best_s8) best_s8 = v;
    cudaEventRecord(e0);
    mma_f16<<<blocks, threads>>>(iters, out);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    cudaEventElapsedTime(&ms, e0, e1);
    v = 2.0 * 16 * 8 * 16 * 4.0 * iters * warps / ms / 1e9;
    if (v > best_f16) best_f16 = v;
  }
  printf("{\"engine\": \"mma.sync m16n8k32 s8->s32\", \"tops\": %.1f}\n", best_s8);
  printf("{\"engine\": \"mma.sync m16n8k16 f16->f32\", \"tflops\": %.1f}\n", best_f16);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}
"""


def engine_rates():
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "mma_sync_rates.cu")
        exe = os.path.join(d, "mma_sync_rates")
        with open(src, "w") as fh:
            fh.write(MMA_SYNC_SRC)
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe, src],
                       check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    for line in out.splitlines():
        print(line, flush=True)


def _time(fn, iters):
    """Device time per call: `iters` calls captured into one CUDA graph and
    replayed, so host-side launch cost (the Python binding's marshalling)
    does not starve the GPU on small shapes."""
    for _ in range(3):
        fn(0)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(iters):
                fn(i)
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    reps = 3
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * iters) * 1e-3


def shape_row(shape, iters, full=True):
    M, K, N = shape.M, shape.K, shape.N
    d = inputs.linear_inputs(shape)
    dev = "cuda"
    w = d["w"].to(dev)
    b = d["bias"].to(dev)
    wq, s_w = i8.quant_weight_perchannel(w)
    w16 = i8.widen_weight_codes(wq)
    # Every set holds its own copy of the weights too: with few tokens the
    # weights are most of the bytes, and one shared copy would stay in L2.
    # The bytes of one call (int8 weights, the smallest) times R exceed 3 x L2.
    per_set = M * K + N * K + M * N * 2
    R = max(2, min(64, -(-3 * 129 * 2**20 // max(per_set, 1))))
    wqs = [wq] + [wq.clone() for _ in range(R - 1)]
    w16s = [w16] + [w16.clone() for _ in range(R - 1)]
    xs = [d["x"].to(dev) for _ in range(R)]
    aqs = [torch.empty(M, K, dtype=torch.int8, device=dev) for _ in range(R)]
    sas = [torch.empty(M, dtype=torch.float32, device=dev) for _ in range(R)]
    ys = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    ws = torch.empty(max(i8.workspace_bytes(M, N, K), 16), dtype=torch.uint8, device=dev)
    for r in range(R):
        i8.quant_act_pertoken(xs[r], aqs[r], sas[r])
    ops = 2.0 * M * N * K
    res = {"shape": shape.name, "M": M, "K": K, "N": N, "l2_sets": R,
           "k_splits": "yes" if i8.workspace_bytes(M, N, K) else "no"}

    def step(wmats):
        def f(i):
            r = i % R
            i8.quant_act_pertoken(xs[r], aqs[r], sas[r])
            i8.gemm_dequant_bias_bf16(aqs[r], sas[r], wmats[r], s_w, b, out=ys[r], workspace=ws)
        return f

    def gemm(wmats):
        def f(i):
            r = i % R
            i8.gemm_dequant_bias_bf16(aqs[r], sas[r], wmats[r], s_w, b, out=ys[r], workspace=ws)
        return f

    for key, fn in (("step_int8_us", step(wqs)), ("gemm_int8_us", gemm(wqs)),
                    ("step_w16_us", step(w16s)), ("gemm_w16_us", gemm(w16s))):
        res[key] = _time(fn, iters) * 1e6
    i8.sync_check()
    res["gemm_int8_tops"] = ops / (res["gemm_int8_us"] * 1e-6) / 1e12
    res["gemm_w16_tops"] = ops / (res["gemm_w16_us"] * 1e-6) / 1e12
    res["step_int8_tops"] = ops / (res["step_int8_us"] * 1e-6) / 1e12
    # the E4M3 arm on the same inputs
    wq8, s_w8 = i8.quant_weight_perchannel_e4m3(w)
    wq8s = [wq8] + [wq8.clone() for _ in range(R - 1)]
    aq8 = [torch.empty(M, K, dtype=torch.float8_e4m3fn, device=dev) for _ in range(R)]
    sa8 = [torch.empty(M, dtype=torch.float32, device=dev) for _ in range(R)]
    for r in range(R):
        i8.quant_act_pertoken_e4m3(xs[r], aq8[r], sa8[r])
    ws8 = torch.empty(max(i8.e4m3_workspace_bytes(M, N, K), 16), dtype=torch.uint8, device=dev)

    def step8(i):
        r = i % R
        i8.quant_act_pertoken_e4m3(xs[r], aq8[r], sa8[r])
        i8.gemm_e4m3_dequant_bias_bf16(aq8[r], sa8[r], wq8s[r], s_w8, b, out=ys[r], workspace=ws8)

    def gemm8(i):
        r = i % R
        i8.gemm_e4m3_dequant_bias_bf16(aq8[r], sa8[r], wq8s[r], s_w8, b, out=ys[r], workspace=ws8)

    res["step_e4m3_us"] = _time(step8, iters) * 1e6
    res["gemm_e4m3_us"] = _time(gemm8, iters) * 1e6
    # the exact path with fp16-held codes (weights widened offline)
    a16 = [torch.empty(M, K, dtype=torch.float16, device=dev) for _ in range(R)]
    for r in range(R):
        i8.quant_act_pertoken_f16codes(xs[r], a16[r], sas[r])
    ws16 = torch.empty(max(i8.f16codes_workspace_bytes(M, N, K), 16), dtype=torch.uint8, device=dev)

    def step16(i):
        r = i % R
        i8.quant_act_pertoken_f16codes(xs[r], a16[r], sas[r])
        i8.gemm_dequant_bias_bf16_f16codes(a16[r], sas[r], w16s[r], s_w, b, out=ys[r], workspace=ws16)

    def gemm16(i):
        r = i % R
        i8.gemm_dequant_bias_bf16_f16codes(a16[r], sas[r], w16s[r], s_w, b, out=ys[r], workspace=ws16)

    res["step_f16codes_us"] = _time(step16, iters) * 1e6
    res["gemm_f16codes_us"] = _time(gemm16, iters) * 1e6
    res["gemm_f16codes_tops"] = ops / (res["gemm_f16codes_us"] * 1e-6) / 1e12
    i8.sync_check()
    res["gemm_e4m3_tflops"] = ops / (res["gemm_e4m3_us"] * 1e-6) / 1e12
    res["e4m3_k_splits"] = "yes" if i8.e4m3_workspace_bytes(M, N, K) else "no"
    if full:
        wts = [w.t()] + [w.clone().t() for _ in range(R - 1)]
        res["torch_bf16_us"] = _time(lambda i: torch.addmm(b, xs[i % R], wts[i % R], out=ys[i % R]),
                                     iters) * 1e6
        del wts
        if M > 16:
            res["torch_int_mm_us"] = _time(lambda i: torch._int_mm(aqs[i % R], wqs[i % R].t()), iters) * 1e6
        def fake(i):
            r = i % R
            a_deq = aqs[r].to(torch.bfloat16) * sas[r].to(torch.bfloat16)[:, None]
            w_deq = wqs[r].to(torch.bfloat16) * s_w.to(torch.bfloat16)[:, None]
            torch.addmm(b, a_deq, w_deq.t(), out=ys[r])
        res["fake_int8_us"] = _time(fake, iters) * 1e6
        res["torch_bf16_tflops"] = ops / (res["torch_bf16_us"] * 1e-6) / 1e12
    print(json.dumps(res), flush=True)


def producer_rates(iters=20):
    """The fused producer-quantizers against the unfused path they replace
    (torch LayerNorm / GELU writing bf16, then the separate quantizer), at the
    DiT inputs: LN at M = 8704, K = 3072 (QKV / out / up) and GELU at M = 8704,
    K = 12288 (down), int8 codes.  Inputs rotate over sets larger than 3 x L2.
    Fused bytes: 2 MK read + MK written + 4 M; unfused: the torch op's 2 MK
    read + 2 MK written, then the quantizer's 3 MK + 4 M."""
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {"hbm_gbs": 6800.0}
    hbm = float(peaks["hbm_gbs"])
    for op, K in (("layernorm", 3072), ("gelu", 12288)):
        M = 8704
        R = max(2, -(-3 * 129 * 2 ** 20 // (M * K * 3)))
        xs = [inputs.activations(M, K, torch.Generator().manual_seed(11 + r)).to("cuda") for r in range(R)]
        qs = [torch.empty(M, K, dtype=torch.int8, device="cuda") for _ in range(R)]
        ss = [torch.empty(M, dtype=torch.float32, device="cuda") for _ in range(R)]
        lib = i8.load()
        vp = ctypes.c_void_p

        def fused(i):
            st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            x, q, s = xs[i % R], qs[i % R], ss[i % R]
            if op == "layernorm":
                rc = lib.i8_layernorm_quant_act_pertoken(vp(x.data_ptr()), M, K, K, ctypes.c_float(1e-6), 0,
                                                         vp(q.data_ptr()), K, vp(s.data_ptr()), None, 0, st)
            else:
                rc = lib.i8_gelu_quant_act_pertoken(vp(x.data_ptr()), M, K, K, 0, vp(q.data_ptr()), K,
                                                    vp(s.data_ptr()), None, 0, st)
            assert rc == 0

        def unfused(i):
            x = xs[i % R]
            y = (torch.nn.functional.layer_norm(x, (K,), eps=1e-6) if op == "layernorm"
                 else torch.nn.functional.gelu(x, approximate="none"))
            i8.quant_act_pertoken(y, q=qs[i % R], s=ss[i % R])

        t_f = _time(fused, iters)
        t_u = _time(unfused, iters)
        b_f = 3.0 * M * K + 4.0 * M
        b_u = 4.0 * M * K + 3.0 * M * K + 4.0 * M
        print(json.dumps({"producer": op, "M": M, "K": K, "codes": "int8",
                          "fused_us": t_f * 1e6, "fused_gbs": b_f / t_f / 1e9,
                          "fused_frac_hbm": b_f / t_f / 1e9 / hbm,
                          "unfused_us": t_u * 1e6, "unfused_gbs": b_u / t_u / 1e9,
                          "speedup": t_u / t_f, "hbm_peak_gbs": hbm}), flush=True)
        del xs, qs, ss
        torch.cuda.empty_cache()


def stack_time(blocks=28, M=8704, iters=5, fused=False, fmt="int8"):
    """Linear-layer time per denoising step of the synthetic 28-block DiT
    stack at 1024px batch 2 (M = 8704): the sum over 112 layers of each
    layer's quantizer and fused GEMM, timed with CUDA events around each
    layer.  Unfused, the glue (LayerNorm, GELU, V slice) runs in torch between
    the timed layers; fused, the LayerNorm / GELU in front of each layer runs
    inside the timed producer-quantizer kernel and only the block-output LN
    stays outside.  step_ms_with_glue is the whole forward either way."""
    from w8a8_int8_quantized_i8_gb300 import dit_stack
    stack = dit_stack.build(blocks=blocks, seed=5, fmt=fmt)
    h = inputs.activations(M, dit_stack.WIDTH, torch.Generator().manual_seed(5)).to("cuda")
    events = []

    def timer(begin):
        ev = torch.cuda.Event(enable_timing=True)
        ev.record()
        events.append(ev)

    dit_stack.forward(stack, h, fused=fused)  # warm-up
    torch.cuda.synchronize()
    lin, tot = [], []
    for _ in range(iters):
        events.clear()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        dit_stack.forward(stack, h, timer=timer, fused=fused)
        e1.record()
        torch.cuda.synchronize()
        lin.append(sum(events[i].elapsed_time(events[i + 1]) for i in range(0, len(events), 2)))
        tot.append(e0.elapsed_time(e1))
    i8.sync_check()
    # whole forward without per-layer events
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        dit_stack.forward(stack, h, fused=fused)
    e1.record()
    torch.cuda.synchronize()
    ops = 2.0 * M * blocks * sum(K * N for _, K, N in dit_stack.LAYERS)
    lin_ms = sorted(lin)[len(lin) // 2]
    print(json.dumps({"stack": f"dit_1024px_b2_{blocks}blocks_M{M}", "codes": fmt,
                      "producers": "fused LN/GELU + quant" if fused else "torch LN/GELU, separate quant",
                      "linear_ms_per_step": lin_ms,
                      "step_ms_with_glue": sorted(tot)[len(tot) // 2],
                      "step_ms_no_events": e0.elapsed_time(e1) / iters, "layers": 4 * blocks,
                      "linear_tops": ops / (lin_ms * 1e-3) / 1e12}), flush=True)
    del stack
    torch.cuda.empty_cache()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--sweep", action="store_true", help="also run the 35-shape sweep")
    ap.add_argument("--iters", type=int, default=30)
    ap.add_argument("--no-engines", action="store_true")
    ap.add_argument("--stack", action="store_true", help="time the 28-block DiT linear stack")
    ap.add_argument("--producers", action="store_true",
                    help="time the fused LayerNorm/GELU + quant kernels against the unfused path")
    ap.add_argument("--no-shapes", action="store_true", help="skip the three DiT layer rows")
    args = ap.parse_args(argv)
    i8.load()
    if not args.no_engines:
        engine_rates()
    if not args.no_shapes:
        for shape in (inputs.QKV_768, inputs.MLP_UP_1024, inputs.MLP_DOWN_1024):
            shape_row(shape, args.iters)
    if args.producers:
        producer_rates()
    if args.sweep:
        for shape in inputs.sweep_shapes():
            shape_row(shape, args.iters, full=True)
    if args.stack:
        for fmt in ("int8", "f16codes", "e4m3"):
            for fused in (False, True):
                stack_time(fused=fused, fmt=fmt)
    return 0


if __name__ == "__main__":
    sys.exit(main())
