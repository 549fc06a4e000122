"""CPU oracle for the W8A8 linear layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never touches it, and it never touches the product path:
the two share no code.

The arithmetic lives in ``i8_oracle.c`` (plain C, fp32 steps in the order the
pages give them); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  bf16 tensors travel as ``uint16`` bit patterns.

Source: "Realizing Native INT8 Compute for Diffusion Transformers on Consumer
GPUs: A Fused INT8 GEMM Kernel for Ideogram 4.0" (arXiv 2606.14598), abstract:
per-token activation and per-channel weight INT8 quantization, an int8 x int8
-> int32 GEMM, and a per-token x per-channel dequantization plus bias epilogue
that emits bf16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "i8_oracle.c")
_HDR = os.path.join(_HERE, "i8_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-fopenmp", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, no intrinsics)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC),
                                              os.path.getmtime(_HDR))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, vp = ctypes.c_int64, ctypes.c_void_p
            lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f32.restype = ctypes.c_float
            lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_bf16.restype = ctypes.c_uint16
            lib.orc_quant_rows.argtypes = [vp, i64, i64, i64, vp, i64, vp]
            lib.orc_quant_rows.restype = ctypes.c_int
            lib.orc_gemm_s32.argtypes = [vp, i64, vp, i64, i64, i64, i64, vp, i64]
            lib.orc_gemm_s32.restype = ctypes.c_int
            lib.orc_dequant_bias.argtypes = [vp, i64, vp, vp, vp, i64, i64, vp, i64]
            lib.orc_dequant_bias.restype = ctypes.c_int
            lib.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
            lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
            lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_f64.restype = ctypes.c_double
            lib.orc_quant_rows_e4m3.argtypes = [vp, i64, i64, i64, vp, i64, vp]
            lib.orc_quant_rows_e4m3.restype = ctypes.c_int
            lib.orc_gemm_e4m3_f64.argtypes = [vp, i64, vp, i64, i64, i64, i64,
                                              ctypes.c_int, vp, i64]
            lib.orc_gemm_e4m3_f64.restype = ctypes.c_int
            lib.orc_dequant_bias_f64acc.argtypes = [vp, i64, vp, vp, vp, i64, i64, vp, i64]
            lib.orc_dequant_bias_f64acc.restype = ctypes.c_int
            lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.orc_f64_to_bf16.restype = ctypes.c_uint16
            lib.orc_layernorm_rows.argtypes = [vp, i64, i64, i64, ctypes.c_double, vp, i64]
            lib.orc_layernorm_rows.restype = ctypes.c_int
            lib.orc_gelu_rows.argtypes = [vp, i64, i64, i64, vp, i64]
            lib.orc_gelu_rows.restype = ctypes.c_int
            lib.orc_num_threads.argtypes = []
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_set_num_threads.argtypes = [ctypes.c_int]
            lib.orc_set_num_threads.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c2d(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    if a.ndim != 2:
        raise ValueError("expected a 2-D array")
    return np.ascontiguousarray(a)


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


def f32_to_bf16_bits(f: float) -> int:
    return int(_load().orc_f32_to_bf16(float(f)))


def bf16_bits_to_f32(b: int) -> float:
    return float(_load().orc_bf16_to_f32(int(b)))


def quant_rows(x_bits):
    """Per-row symmetric INT8 quantization of a bf16 matrix (uint16 bits).

    Returns ``(q int8 [rows,K], scale float32 [rows])``.
    """
    x = _c2d(x_bits, np.uint16)
    rows, K = x.shape
    q = np.zeros((rows, K), dtype=np.int8)
    s = np.zeros((rows,), dtype=np.float32)
    rc = _load().orc_quant_rows(_ptr(x), rows, K, K, _ptr(q), K, _ptr(s))
    if rc != 0:
        raise ValueError("orc_quant_rows rejected its arguments")
    return q, s


def gemm_s32(a, w) -> np.ndarray:
    """int32 ``a @ w.T`` for int8 ``a [M,K]`` and ``w [N,K]``."""
    a = _c2d(a, np.int8)
    w = _c2d(w, np.int8)
    M, K = a.shape
    N, K2 = w.shape
    if K != K2:
        raise ValueError("K mismatch")
    c = np.zeros((M, N), dtype=np.int32)
    rc = _load().orc_gemm_s32(_ptr(a), K, _ptr(w), K, M, N, K, _ptr(c), N)
    if rc != 0:
        raise ValueError("orc_gemm_s32 rejected its arguments")
    return c


def dequant_bias(acc, s_a, s_w, bias_bits) -> np.ndarray:
    """bf16 bits of ``acc * s_a[:,None] * s_w[None,:] + bias`` (see the C file)."""
    c = _c2d(acc, np.int32)
    M, N = c.shape
    sa = np.ascontiguousarray(s_a, dtype=np.float32)
    sw = np.ascontiguousarray(s_w, dtype=np.float32)
    if sa.shape != (M,) or sw.shape != (N,):
        raise ValueError("scale shapes")
    b = None
    if bias_bits is not None:
        b = np.ascontiguousarray(bias_bits)
        if b.dtype != np.uint16 or b.shape != (N,):
            raise ValueError("bias must be uint16 bf16 bits of shape [N]")
    y = np.zeros((M, N), dtype=np.uint16)
    rc = _load().orc_dequant_bias(_ptr(c), N, _ptr(sa), _ptr(sw), _ptr(b), M, N,
                                  _ptr(y), N)
    if rc != 0:
        raise ValueError("orc_dequant_bias rejected its arguments")
    return y


def linear(x_bits, w_bits, bias_bits):
    """The whole path: quantize X per token and W per channel, GEMM, epilogue.

    Returns a dict with ``aq, s_a, wq, s_w, acc, y`` (y as bf16 bits).
    """
    aq, s_a = quant_rows(x_bits)
    wq, s_w = quant_rows(w_bits)
    acc = gemm_s32(aq, wq)
    y = dequant_bias(acc, s_a, s_w, bias_bits)
    return dict(aq=aq, s_a=s_a, wq=wq, s_w=s_w, acc=acc, y=y)


# ---------------------------------------------------------------------- FP8
# The E4M3 arm (see the FP8 section of i8_oracle.h for the reading): the same
# per-row symmetric scheme with s = absmax / 448 and E4M3 codes, an exact
# fp64 GEMM over the codes, and the same fp32 epilogue steps.

def f32_to_e4m3_bits(f: float) -> int:
    return int(_load().orc_f32_to_e4m3(float(f)))


def e4m3_bits_to_f64(b: int) -> float:
    return float(_load().orc_e4m3_to_f64(int(b)))


def quant_rows_e4m3(x_bits):
    """Per-row E4M3 quantization of a bf16 matrix (uint16 bits).

    Returns ``(q uint8 [rows,K] E4M3 bit patterns, scale float32 [rows])``.
    """
    x = _c2d(x_bits, np.uint16)
    rows, K = x.shape
    q = np.zeros((rows, K), dtype=np.uint8)
    s = np.zeros((rows,), dtype=np.float32)
    rc = _load().orc_quant_rows_e4m3(_ptr(x), rows, K, K, _ptr(q), K, _ptr(s))
    if rc != 0:
        raise ValueError("orc_quant_rows_e4m3 rejected its arguments")
    return q, s


def gemm_e4m3_f64(a, w, absval: bool = False) -> np.ndarray:
    """Exact fp64 ``a @ w.T`` over E4M3 codes (``|a| @ |w|.T`` if absval)."""
    a = _c2d(a, np.uint8)
    w = _c2d(w, np.uint8)
    M, K = a.shape
    N, K2 = w.shape
    if K != K2:
        raise ValueError("K mismatch")
    c = np.zeros((M, N), dtype=np.float64)
    rc = _load().orc_gemm_e4m3_f64(_ptr(a), K, _ptr(w), K, M, N, K,
                                   1 if absval else 0, _ptr(c), N)
    if rc != 0:
        raise ValueError("orc_gemm_e4m3_f64 rejected its arguments")
    return c


def dequant_bias_f64acc(acc, s_a, s_w, bias_bits) -> np.ndarray:
    """bf16 bits of ``fl32(acc) * s_a * s_w + bias`` with fp32 steps."""
    c = _c2d(acc, np.float64)
    M, N = c.shape
    sa = np.ascontiguousarray(s_a, dtype=np.float32)
    sw = np.ascontiguousarray(s_w, dtype=np.float32)
    if sa.shape != (M,) or sw.shape != (N,):
        raise ValueError("scale shapes")
    b = None
    if bias_bits is not None:
        b = np.ascontiguousarray(bias_bits)
        if b.dtype != np.uint16 or b.shape != (N,):
            raise ValueError("bias must be uint16 bf16 bits of shape [N]")
    y = np.zeros((M, N), dtype=np.uint16)
    rc = _load().orc_dequant_bias_f64acc(_ptr(c), N, _ptr(sa), _ptr(sw), _ptr(b),
                                         M, N, _ptr(y), N)
    if rc != 0:
        raise ValueError("orc_dequant_bias_f64acc rejected its arguments")
    return y


def linear_e4m3(x_bits, w_bits, bias_bits):
    """The E4M3 path: per-row E4M3 quantization of X and W, the exact GEMM
    over the codes, and the epilogue.  Returns ``aq, s_a, wq, s_w, acc, y``
    (acc exact in fp64, y as bf16 bits)."""
    aq, s_a = quant_rows_e4m3(x_bits)
    wq, s_w = quant_rows_e4m3(w_bits)
    acc = gemm_e4m3_f64(aq, wq)
    y = dequant_bias_f64acc(acc, s_a, s_w, bias_bits)
    return dict(aq=aq, s_a=s_a, wq=wq, s_w=s_w, acc=acc, y=y)


# ---------------------------------------------------------------------- fused
# The producer of a linear layer's input (LayerNorm without affine, or GELU),
# in fp64 with one rounding to bf16, followed by the per-row quantizer of that
# bf16 row (see the fused section of i8_oracle.h).

def f64_to_bf16_bits(v: float) -> int:
    return int(_load().orc_f64_to_bf16(float(v)))


def layernorm_rows(x_bits, eps: float = 1e-6) -> np.ndarray:
    """bf16 bits of the row-wise LayerNorm (no affine) of a bf16 matrix."""
    x = _c2d(x_bits, np.uint16)
    rows, K = x.shape
    y = np.zeros((rows, K), dtype=np.uint16)
    if _load().orc_layernorm_rows(_ptr(x), rows, K, K, float(eps), _ptr(y), K) != 0:
        raise ValueError("orc_layernorm_rows rejected its arguments")
    return y


def gelu_rows(x_bits) -> np.ndarray:
    """bf16 bits of GELU (erf form) of a bf16 matrix."""
    x = _c2d(x_bits, np.uint16)
    rows, K = x.shape
    y = np.zeros((rows, K), dtype=np.uint16)
    if _load().orc_gelu_rows(_ptr(x), rows, K, K, _ptr(y), K) != 0:
        raise ValueError("orc_gelu_rows rejected its arguments")
    return y


def producer_quant_rows(x_bits, op: str, fmt: str = "int8", eps: float = 1e-6):
    """LayerNorm (op="layernorm") or GELU (op="gelu") then the per-row
    quantizer ("int8" or "e4m3").  Returns ``(y bf16 bits, q, scale)``."""
    y = layernorm_rows(x_bits, eps) if op == "layernorm" else gelu_rows(x_bits)
    q, s = quant_rows(y) if fmt == "int8" else quant_rows_e4m3(y)
    return y, q, s
