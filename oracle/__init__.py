"""CPU oracle for the compensated-FP32 projection — TEST INFRASTRUCTURE ONLY.

A ctypes front end for ``oracle.c``: plain, slow, obviously correct CPU code that
the CUDA library is checked against.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package; the CUDA library never
does, and this package never imports the library.

The method (laya.cpp, "docs/vulkan.md", paragraphs on compensated FP32 and on
the split/merge dispatches): each FP32 input x becomes hi = fp16_rne(x) and
lo = fp16_rne((x - hi) * 1024), both products against the exact FP16 weights
are accumulated in FP32, and the results are combined in FP32 as
y = acc_hi + acc_lo * 2^-10.

Arrays are numpy; FP16 values travel as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-pthread", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, plain C11)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, c_int = ctypes.c_int64, ctypes.c_int
        vp = ctypes.c_void_p
        lib.oracle_fp16_rne.argtypes = [ctypes.c_double]
        lib.oracle_fp16_rne.restype = ctypes.c_uint16
        lib.oracle_fp16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_value.restype = ctypes.c_double
        lib.oracle_default_threads.argtypes = []
        lib.oracle_default_threads.restype = c_int
        lib.oracle_split.argtypes = [vp, vp, vp, i64, c_int]
        lib.oracle_merge.argtypes = [vp, vp, vp, i64, c_int]
        lib.oracle_epilogue.argtypes = [vp, vp, vp, vp, i64, i64, c_int]
        lib.oracle_gelu.argtypes = [ctypes.c_double]
        lib.oracle_gelu.restype = ctypes.c_double
        for name in ("oracle_gemm_comp", "oracle_gemm_true", "oracle_gemm_cast", "oracle_gemm_den"):
            getattr(lib, name).argtypes = [vp, vp, i64, i64, i64, vp, vp, i64, vp, c_int]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def default_threads() -> int:
    """Host threads the oracle uses when not told otherwise (all online cores)."""
    return int(_load().oracle_default_threads())


def fp16_rne(v: float) -> int:
    """binary16 round-to-nearest-even of one real value (given as a double), as bits."""
    return int(_load().oracle_fp16_rne(float(v)))


def fp16_value(h: int) -> float:
    """Exact value of a binary16 bit pattern."""
    return float(_load().oracle_fp16_value(int(h) & 0xFFFF))


def split(x: np.ndarray, threads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """hi, lo (uint16 bit planes, same shape as x) for a float32 array x."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    hi = np.empty(x.shape, np.uint16)
    lo = np.empty(x.shape, np.uint16)
    _load().oracle_split(_ptr(x), _ptr(hi), _ptr(lo), x.size, threads)
    return hi, lo


def merge(acc_hi: np.ndarray, acc_lo: np.ndarray, threads: int = 0) -> np.ndarray:
    """y = acc_hi + acc_lo * 2^-10 in binary32 (product then sum, each rounded)."""
    a = np.ascontiguousarray(acc_hi, dtype=np.float32)
    b = np.ascontiguousarray(acc_lo, dtype=np.float32)
    if a.shape != b.shape:
        raise ValueError("acc_hi and acc_lo differ in shape")
    y = np.empty(a.shape, np.float32)
    _load().oracle_merge(_ptr(a), _ptr(b), _ptr(y), a.size, threads)
    return y


def _gemm(name: str, x, W, rows, cols, threads: int, out_dtype):
    x = np.ascontiguousarray(x, dtype=np.float32)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    if x.ndim != 2 or W.ndim != 2 or x.shape[1] != W.shape[1]:
        raise ValueError("x must be [M, K] float32 and W [N, K] binary16 bits")
    M, K = x.shape
    N = W.shape[0]
    fn = getattr(_load(), name)
    if rows is None:
        out = np.empty((M, N), out_dtype)
        fn(_ptr(x), _ptr(W), M, N, K, None, None, 0, _ptr(out), threads)
        return out
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape or r.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    if r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise ValueError("sample index out of range")
    out = np.empty(r.shape, out_dtype)
    fn(_ptr(x), _ptr(W), M, N, K, _ptr(r), _ptr(c), r.size, _ptr(out), threads)
    return out


def gemm_comp(x, W, rows=None, cols=None, threads: int = 0) -> np.ndarray:
    """The method's result, sums in FP64: fp32(sum hi*w + 2^-10 * sum lo*w)."""
    return _gemm("oracle_gemm_comp", x, W, rows, cols, threads, np.float32)


def gemm_true(x, W, rows=None, cols=None, threads: int = 0) -> np.ndarray:
    """The exact product of the FP32 input, sums in FP64: fp32(sum x*w)."""
    return _gemm("oracle_gemm_true", x, W, rows, cols, threads, np.float32)


def gemm_cast(x, W, rows=None, cols=None, threads: int = 0) -> np.ndarray:
    """A single FP16 cast of x, sums in FP64: fp32(sum fp16(x)*w)."""
    return _gemm("oracle_gemm_cast", x, W, rows, cols, threads, np.float32)


def gemm_den(x, W, rows=None, cols=None, threads: int = 0) -> np.ndarray:
    """Error scale per output: sum |x|*|w| (float64)."""
    return _gemm("oracle_gemm_den", x, W, rows, cols, threads, np.float64)


def gelu(g: float) -> float:
    """The exact GELU g * Phi(g) in double."""
    return float(_load().oracle_gelu(float(g)))


def epilogue(y, bias=None, gate=None, threads: int = 0) -> np.ndarray:
    """out = gelu(gate) * (y + bias) per element of y [M, N], bias [N] and gate
    [M, N] optional; double arithmetic, rounded once to binary32."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    if y.ndim != 2:
        raise ValueError("y must be [M, N]")
    M, N = y.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    g = None if gate is None else np.ascontiguousarray(gate, dtype=np.float32)
    if b is not None and b.shape != (N,):
        raise ValueError("bias must be [N]")
    if g is not None and g.shape != (M, N):
        raise ValueError("gate must be [M, N]")
    out = np.empty((M, N), np.float32)
    _load().oracle_epilogue(_ptr(y), None if b is None else _ptr(b), None if g is None else _ptr(g), _ptr(out), M, N,
                            threads)
    return out

