"""Thin Python binding over libi8 (include/i8.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
checks tensor dtypes/devices/shapes, allocates outputs with torch (the
library itself allocates nothing), passes raw device pointers and the
current CUDA stream, and turns status codes into exceptions.  There is no
fallback: if libi8.so is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS = {
    0: "I8_OK", 1: "I8_ERR_INVALID_ARG", 2: "I8_ERR_ALIGNMENT", 3: "I8_ERR_UNSUPPORTED",
    4: "I8_ERR_WORKSPACE", 5: "I8_ERR_CUDA", 6: "I8_ERR_DEVICE_TIMEOUT",
}
OPTIONS = {"chunk_k": 1, "force_splits": 2, "max_ctas": 3, "tile_n": 4, "quant_vpl": 5, "cta_pair": 6,
           "skinny_max_m": 7, "pdl": 8, "quant_rows": 9, "stream_k": 10, "nvtx": 11,
           "pair_stage_k": 12, "raster": 13}


ROUTES = {"int8": 0, "w16": 1, "f16codes": 2, "e4m3": 3}
KERNELS = {0: "skinny", 1: "tile", 2: "pair", 3: "pair_stream_k", 4: "direct"}


class PlanInfo(ctypes.Structure):
    """i8_plan_info of include/i8.h."""
    _fields_ = [("kernel", ctypes.c_int32), ("tile_m", ctypes.c_int32),
                ("tile_n", ctypes.c_int32), ("num_m", ctypes.c_int32),
                ("num_n", ctypes.c_int32), ("block_k", ctypes.c_int32),
                ("total_kb", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("kb_per_split", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("n_fastest", ctypes.c_int32), ("ws_bytes", ctypes.c_int64),
                ("model_us", ctypes.c_double), ("sk_waves", ctypes.c_int32),
                ("sk_pairs", ctypes.c_int32)]


class I8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


def header_functions() -> list[str]:
    """Names of the functions declared in include/i8.h."""
    hdr = os.path.join(_build.ROOT, "include", "i8.h")
    with open(hdr) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\**\s+\**(i8_[a-z0-9_]+)\s*\(",
                      text, flags=re.M)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libi8.so (building it first if it is stale).  Raises on failure."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        if path is None:
            path = _build.build()
        if not os.path.exists(path):
            raise OSError(f"libi8 not found at {path}")
        lib = ctypes.CDLL(path)
        i64, vp, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        st = ctypes.c_int
        sigs = {
            "i8_status_string": ([st], ctypes.c_char_p),
            "i8_version": ([], ctypes.c_char_p),
            "i8_quant_weight_perchannel": ([vp, i64, i64, i64, vp, i64, vp, vp], st),
            "i8_quant_act_pertoken": ([vp, i64, i64, i64, vp, i64, vp, vp], st),
            "i8_gemm_workspace_bytes": ([i64, i64, i64], sz),
            "i8_gemm_int32": ([vp, vp, i64, i64, i64, vp, i64, vp, sz, vp], st),
            "i8_gemm_dequant_bias_bf16": ([vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp, sz, vp], st),
            "i8_widen_weight_codes": ([vp, i64, i64, vp, vp], st),
            "i8_gemm_dequant_bias_bf16_w16": ([vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp, sz, vp], st),
            "i8_set_option": ([ctypes.c_int, i64], st),
            "i8_get_option": ([ctypes.c_int, ctypes.POINTER(ctypes.c_int64)], st),
            "i8_gemm_dequant_bias_bf16_noalloc": ([vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp], st),
            "i8_quant_weight_perchannel_e4m3": ([vp, i64, i64, i64, vp, i64, vp, vp], st),
            "i8_quant_act_pertoken_e4m3": ([vp, i64, i64, i64, vp, i64, vp, vp], st),
            "i8_gemm_e4m3_workspace_bytes": ([i64, i64, i64], sz),
            "i8_gemm_e4m3_f32": ([vp, vp, i64, i64, i64, vp, i64, vp, sz, vp], st),
            "i8_gemm_e4m3_dequant_bias_bf16": ([vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp, sz,
                                                vp], st),
            "i8_quant_act_pertoken_f16codes": ([vp, i64, i64, i64, vp, i64, vp, vp], st),
            "i8_gemm_f16codes_workspace_bytes": ([i64, i64, i64], sz),
            "i8_gemm_int32_f16codes": ([vp, vp, i64, i64, i64, vp, i64, vp, sz, vp], st),
            "i8_gemm_dequant_bias_bf16_f16codes": ([vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp,
                                                    sz, vp], st),
            "i8_layernorm_quant_act_pertoken": ([vp, i64, i64, i64, ctypes.c_float, ctypes.c_int,
                                                 vp, i64, vp, vp, i64, vp], st),
            "i8_gelu_quant_act_pertoken": ([vp, i64, i64, i64, ctypes.c_int, vp, i64, vp, vp, i64,
                                            vp], st),
            "i8_sync_check": ([vp], st),
            "i8_selftest_timeout": ([ctypes.c_int, vp], st),
            "i8_plan_query": ([i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, sz, ctypes.POINTER(PlanInfo)], st),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        if path == _build.LIB:
            _lib = lib
        return lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise I8Error(status, what)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, dtype, name: str, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _quant(fn_name: str, x: torch.Tensor, q=None, s=None):
    _need(x, torch.bfloat16, "x", 2)
    R, K = x.shape
    if q is None:
        q = torch.empty((R, K), dtype=torch.int8, device=x.device)
    if s is None:
        s = torch.empty((R,), dtype=torch.float32, device=x.device)
    _need(q, torch.int8, "q", 2)
    _need(s, torch.float32, "s", 1)
    if tuple(q.shape) != (R, K) or s.shape[0] != R:
        raise ValueError("output shape")
    lib = load()
    with torch.cuda.device(x.device):
        _check(getattr(lib, fn_name)(_ptr(x), R, K, K, _ptr(q), K, _ptr(s), _stream(x)), fn_name)
    return q, s


def quant_act_pertoken(x: torch.Tensor, q=None, s=None):
    """bf16 [M,K] -> (int8 codes [M,K], fp32 per-token scales [M])."""
    return _quant("i8_quant_act_pertoken", x, q, s)


def quant_weight_perchannel(w: torch.Tensor, q=None, s=None):
    """bf16 [N,K] -> (int8 codes [N,K], fp32 per-channel scales [N])."""
    return _quant("i8_quant_weight_perchannel", w, q, s)


def widen_weight_codes(wq: torch.Tensor) -> torch.Tensor:
    """int8 weight codes [N,K] -> the same integers as fp16 [N,K] (exact)."""
    _need(wq, torch.int8, "wq", 2)
    N, K = wq.shape
    w16 = torch.empty((N, K), dtype=torch.float16, device=wq.device)
    with torch.cuda.device(wq.device):
        _check(load().i8_widen_weight_codes(_ptr(wq), N, K, _ptr(w16), _stream(wq)),
               "i8_widen_weight_codes")
    return w16


def workspace_bytes(M: int, N: int, K: int) -> int:
    """Workspace bytes the int8-code GEMMs need for this shape (0: none): the
    larger of the int8-weight and pre-widened-weight plans."""
    return int(load().i8_gemm_workspace_bytes(M, N, K))


def _workspace(M, N, K, device, workspace):
    need = workspace_bytes(M, N, K)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def gemm_int32(aq: torch.Tensor, wq: torch.Tensor, out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Exact int32 accumulators aq @ wq.T (int8 [M,K] x int8 [N,K])."""
    _need(aq, torch.int8, "aq", 2)
    _need(wq, torch.int8, "wq", 2)
    M, K = aq.shape
    N = wq.shape[0]
    if wq.shape[1] != K:
        raise ValueError("K mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=aq.device)
    _need(out, torch.int32, "out", 2)
    ws, wsb = _workspace(M, N, K, aq.device, workspace)
    with torch.cuda.device(aq.device):
        _check(load().i8_gemm_int32(_ptr(aq), _ptr(wq), M, N, K, _ptr(out), out.stride(0),
                                    _ptr(ws), wsb, _stream(aq)), "i8_gemm_int32")
    return out


def gemm_dequant_bias_bf16(aq, s_a, wq, s_w, bias=None, out=None, workspace=None):
    """Fused W8A8 GEMM: bf16(acc * s_a[m] * s_w[n] + bias[n]).

    ``wq`` is either the int8 codes [N,K] or their fp16-widened copy
    (``widen_weight_codes``); the result is the same either way.
    """
    _need(aq, torch.int8, "aq", 2)
    _need(s_a, torch.float32, "s_a", 1)
    _need(s_w, torch.float32, "s_w", 1)
    wide = isinstance(wq, torch.Tensor) and wq.dtype == torch.float16
    _need(wq, torch.float16 if wide else torch.int8, "wq", 2)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = aq.shape
    N = wq.shape[0]
    if wq.shape[1] != K or s_a.shape[0] != M or s_w.shape[0] != N:
        raise ValueError("shape mismatch")
    if bias is not None and bias.shape[0] != N:
        raise ValueError("bias shape")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    _need(out, torch.bfloat16, "out", 2)
    ws, wsb = _workspace(M, N, K, aq.device, workspace)
    fn = "i8_gemm_dequant_bias_bf16_w16" if wide else "i8_gemm_dequant_bias_bf16"
    with torch.cuda.device(aq.device):
        _check(getattr(load(), fn)(_ptr(aq), _ptr(s_a), _ptr(wq), _ptr(s_w), _ptr(bias), M, N, K,
                                   _ptr(out), out.stride(0), _ptr(ws), wsb, _stream(aq)), fn)
    return out


def linear(x, wq, s_w, bias=None, out=None, workspace=None):
    """The whole W8A8 linear layer: per-token quant of x, then the fused GEMM."""
    aq, s_a = quant_act_pertoken(x)
    return gemm_dequant_bias_bf16(aq, s_a, wq, s_w, bias, out=out, workspace=workspace)


# ---------------------------------------------------------------------- E4M3
# The 8-bit floating-point arm: per-row E4M3 codes (s = absmax / 448) and the
# fused E4M3 GEMM with the same epilogue.  Codes are float8_e4m3fn tensors
# (uint8 tensors holding the same bit patterns are accepted too).

def _codes(t: torch.Tensor, name: str) -> torch.Tensor:
    if isinstance(t, torch.Tensor) and t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    _need(t, torch.uint8, name, 2)
    return t


def _quant_e4m3(fn_name: str, x: torch.Tensor, q=None, s=None):
    _need(x, torch.bfloat16, "x", 2)
    R, K = x.shape
    if q is None:
        q = torch.empty((R, K), dtype=torch.float8_e4m3fn, device=x.device)
    if s is None:
        s = torch.empty((R,), dtype=torch.float32, device=x.device)
    qb = _codes(q, "q")
    _need(s, torch.float32, "s", 1)
    if tuple(qb.shape) != (R, K) or s.shape[0] != R:
        raise ValueError("output shape")
    lib = load()
    with torch.cuda.device(x.device):
        _check(getattr(lib, fn_name)(_ptr(x), R, K, K, _ptr(qb), K, _ptr(s), _stream(x)), fn_name)
    return q, s


def quant_act_pertoken_e4m3(x: torch.Tensor, q=None, s=None):
    """bf16 [M,K] -> (E4M3 codes [M,K], fp32 per-token scales [M])."""
    return _quant_e4m3("i8_quant_act_pertoken_e4m3", x, q, s)


def quant_weight_perchannel_e4m3(w: torch.Tensor, q=None, s=None):
    """bf16 [N,K] -> (E4M3 codes [N,K], fp32 per-channel scales [N])."""
    return _quant_e4m3("i8_quant_weight_perchannel_e4m3", w, q, s)


def e4m3_workspace_bytes(M: int, N: int, K: int) -> int:
    """Workspace bytes the E4M3 GEMMs need for this shape (0: none)."""
    return int(load().i8_gemm_e4m3_workspace_bytes(M, N, K))


def _e4m3_workspace(M, N, K, device, workspace):
    need = e4m3_workspace_bytes(M, N, K)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def gemm_e4m3_f32(aq, wq, out=None, workspace=None) -> torch.Tensor:
    """fp32 tensor-core accumulators aq @ wq.T over E4M3 codes (for checking)."""
    a = _codes(aq, "aq")
    w = _codes(wq, "wq")
    M, K = a.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("K mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=a.device)
    _need(out, torch.float32, "out", 2)
    ws, wsb = _e4m3_workspace(M, N, K, a.device, workspace)
    with torch.cuda.device(a.device):
        _check(load().i8_gemm_e4m3_f32(_ptr(a), _ptr(w), M, N, K, _ptr(out), out.stride(0),
                                       _ptr(ws), wsb, _stream(a)), "i8_gemm_e4m3_f32")
    return out


def gemm_e4m3_dequant_bias_bf16(aq, s_a, wq, s_w, bias=None, out=None, workspace=None):
    """Fused E4M3 GEMM: bf16(acc * s_a[m] * s_w[n] + bias[n])."""
    a = _codes(aq, "aq")
    w = _codes(wq, "wq")
    _need(s_a, torch.float32, "s_a", 1)
    _need(s_w, torch.float32, "s_w", 1)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = a.shape
    N = w.shape[0]
    if w.shape[1] != K or s_a.shape[0] != M or s_w.shape[0] != N:
        raise ValueError("shape mismatch")
    if bias is not None and bias.shape[0] != N:
        raise ValueError("bias shape")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _need(out, torch.bfloat16, "out", 2)
    ws, wsb = _e4m3_workspace(M, N, K, a.device, workspace)
    fn = "i8_gemm_e4m3_dequant_bias_bf16"
    with torch.cuda.device(a.device):
        _check(getattr(load(), fn)(_ptr(a), _ptr(s_a), _ptr(w), _ptr(s_w), _ptr(bias), M, N, K,
                                   _ptr(out), out.stride(0), _ptr(ws), wsb, _stream(a)), fn)
    return out


def linear_e4m3(x, wq, s_w, bias=None, out=None, workspace=None):
    """The E4M3 linear layer: per-token E4M3 quant of x, then the fused GEMM."""
    aq, s_a = quant_act_pertoken_e4m3(x)
    return gemm_e4m3_dequant_bias_bf16(aq, s_a, wq, s_w, bias, out=out, workspace=workspace)


# ---------------------------------------------------------------------- fp16 codes
# The exact W8A8 product with the int8 codes held as fp16 values: the
# quantizer writes them, weights come from widen_weight_codes, and the GEMM
# feeds both to the tensor core without on-chip widening.  Results are
# identical to the int8-code calls.

def quant_act_pertoken_f16codes(x: torch.Tensor, q=None, s=None):
    """bf16 [M,K] -> (int8 codes as fp16 values [M,K], fp32 per-token scales [M])."""
    _need(x, torch.bfloat16, "x", 2)
    R, K = x.shape
    if q is None:
        q = torch.empty((R, K), dtype=torch.float16, device=x.device)
    if s is None:
        s = torch.empty((R,), dtype=torch.float32, device=x.device)
    _need(q, torch.float16, "q", 2)
    _need(s, torch.float32, "s", 1)
    with torch.cuda.device(x.device):
        _check(load().i8_quant_act_pertoken_f16codes(_ptr(x), R, K, K, _ptr(q), K, _ptr(s),
                                                     _stream(x)), "i8_quant_act_pertoken_f16codes")
    return q, s


def f16codes_workspace_bytes(M: int, N: int, K: int) -> int:
    """Workspace bytes the fp16-held-code GEMMs need for this shape (0: none)."""
    return int(load().i8_gemm_f16codes_workspace_bytes(M, N, K))


def _f16_workspace(M, N, K, device, workspace):
    need = f16codes_workspace_bytes(M, N, K)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def gemm_int32_f16codes(a16, w16, out=None, workspace=None) -> torch.Tensor:
    """Exact int32 accumulators from fp16 code values ([M,K] x [N,K])."""
    _need(a16, torch.float16, "a16", 2)
    _need(w16, torch.float16, "w16", 2)
    M, K = a16.shape
    N = w16.shape[0]
    if w16.shape[1] != K:
        raise ValueError("K mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=a16.device)
    _need(out, torch.int32, "out", 2)
    ws, wsb = _f16_workspace(M, N, K, a16.device, workspace)
    with torch.cuda.device(a16.device):
        _check(load().i8_gemm_int32_f16codes(_ptr(a16), _ptr(w16), M, N, K, _ptr(out),
                                             out.stride(0), _ptr(ws), wsb, _stream(a16)),
               "i8_gemm_int32_f16codes")
    return out


def gemm_dequant_bias_bf16_f16codes(a16, s_a, w16, s_w, bias=None, out=None, workspace=None):
    """The fused GEMM from fp16 code values: bf16(acc * s_a[m] * s_w[n] + bias[n])."""
    _need(a16, torch.float16, "a16", 2)
    _need(w16, torch.float16, "w16", 2)
    _need(s_a, torch.float32, "s_a", 1)
    _need(s_w, torch.float32, "s_w", 1)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = a16.shape
    N = w16.shape[0]
    if w16.shape[1] != K or s_a.shape[0] != M or s_w.shape[0] != N:
        raise ValueError("shape mismatch")
    if bias is not None and bias.shape[0] != N:
        raise ValueError("bias shape")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a16.device)
    _need(out, torch.bfloat16, "out", 2)
    ws, wsb = _f16_workspace(M, N, K, a16.device, workspace)
    fn = "i8_gemm_dequant_bias_bf16_f16codes"
    with torch.cuda.device(a16.device):
        _check(getattr(load(), fn)(_ptr(a16), _ptr(s_a), _ptr(w16), _ptr(s_w), _ptr(bias), M, N, K,
                                   _ptr(out), out.stride(0), _ptr(ws), wsb, _stream(a16)), fn)
    return out


def linear_f16codes(x, w16, s_w, bias=None, out=None, workspace=None):
    """The W8A8 layer with fp16-held codes: quantize x, then the fused GEMM."""
    a16, s_a = quant_act_pertoken_f16codes(x)
    return gemm_dequant_bias_bf16_f16codes(a16, s_a, w16, s_w, bias, out=out, workspace=workspace)


# ---------------------------------------------------------------------- fused producers
# LayerNorm (no affine) or GELU of each row, then the per-row quantizer of the
# bf16 result, in one kernel: the codes of the next linear layer's input
# without writing and re-reading that input in bf16.

_FMT = {"int8": (0, torch.int8), "e4m3": (1, torch.float8_e4m3fn), "f16codes": (2, torch.float16)}


def _producer(fn_name, x, extra, fmt, want_y):
    # x may be a row-strided view (e.g. a column slice of a wider output):
    # unit stride along K, any row stride the library accepts
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2:
        raise TypeError("x must be a 2-D bf16 CUDA tensor")
    if x.shape[1] > 1 and x.stride(1) != 1:
        raise ValueError("x must have unit stride along K")
    ldx = x.stride(0) if x.shape[0] > 1 else x.shape[1]
    if ldx < x.shape[1]:
        raise ValueError("x rows overlap")
    if fmt not in _FMT:
        raise ValueError(f"fmt must be one of {sorted(_FMT)}")
    code, dtype = _FMT[fmt]
    R, K = x.shape
    q = torch.empty((R, K), dtype=dtype, device=x.device)
    s = torch.empty((R,), dtype=torch.float32, device=x.device)
    y = torch.empty((R, K), dtype=torch.bfloat16, device=x.device) if want_y else None
    lib = load()
    with torch.cuda.device(x.device):
        _check(getattr(lib, fn_name)(_ptr(x), R, K, ldx, *extra, code, _ptr(q), K, _ptr(s), _ptr(y),
                                     K if want_y else 0, _stream(x)), fn_name)
    return (q, s, y) if want_y else (q, s)


def layernorm_quant_act_pertoken(x: torch.Tensor, eps: float = 1e-6, fmt: str = "int8",
                                 want_y: bool = False):
    """bf16 [M,K] -> codes of LayerNorm(x) (no affine) per token, with scales
    (and the bf16 LayerNorm output when ``want_y``)."""
    return _producer("i8_layernorm_quant_act_pertoken", x, (ctypes.c_float(eps),), fmt, want_y)


def gelu_quant_act_pertoken(x: torch.Tensor, fmt: str = "int8", want_y: bool = False):
    """bf16 [M,K] -> codes of GELU(x) (erf form) per token, with scales (and
    the bf16 GELU output when ``want_y``)."""
    return _producer("i8_gelu_quant_act_pertoken", x, (), fmt, want_y)


def set_option(name: str, value: int) -> None:
    """Set a process-wide tuning option by name (the keys of OPTIONS, which
    mirror i8_option in include/i8.h)."""
    _check(load().i8_set_option(OPTIONS[name], int(value)), f"i8_set_option({name})")


def get_option(name: str) -> int:
    """Current value of a tuning option by name."""
    v = ctypes.c_int64(0)
    _check(load().i8_get_option(OPTIONS[name], ctypes.byref(v)), f"i8_get_option({name})")
    return int(v.value)


def plan_query(M: int, N: int, K: int, route: str = "int8", sms: int = 0, pairs: int = 0,
               skinny_slots: int = 0, ws_cap: int = 0) -> dict:
    """The launch plan the route's GEMM calls would choose for an M x N x K
    shape (i8_plan_query).  With sms > 0 the machine is described by hand and
    no GPU is needed; sms = 0 uses the current device.  Returns the fields of
    i8_plan_info, with ``kernel`` as a name (KERNELS)."""
    info = PlanInfo()
    _check(load().i8_plan_query(int(M), int(N), int(K), ROUTES[route], int(sms), int(pairs),
                                int(skinny_slots), int(ws_cap), ctypes.byref(info)),
           "i8_plan_query")
    out = {name: getattr(info, name) for name, _ in PlanInfo._fields_}
    out["kernel"] = KERNELS[out["kernel"]]
    return out


def sync_check(device=None) -> None:
    """Synchronize the current stream and raise if a kernel recorded an error."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        s = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
        _check(load().i8_sync_check(s), "i8_sync_check")
