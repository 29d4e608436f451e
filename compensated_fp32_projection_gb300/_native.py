"""ctypes binding of ``libcompfp32.so`` (the C ABI in include/compfp32.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  The library is loaded on first use; if it has not been built the call
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcompfp32.so")

COMP_OK = 0
COMP_ERR_INVALID_VALUE = 1
COMP_ERR_MISALIGNED = 2  # reserved, never returned
COMP_ERR_UNSUPPORTED_DEVICE = 3
COMP_ERR_LAUNCH = 4
COMP_ERR_TIMEOUT = 5
COMP_ERR_CUDA = 6

# Every symbol the header declares, with its ctypes signature.
_i64, _int, _u32, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_void_p
SIGNATURES = {
    "comp_split_f32": (_int, [_vp, _vp, _vp, _i64, _vp]),
    "comp_merge_f32": (_int, [_vp, _vp, _vp, _i64, _vp]),
    "comp_gemm_f32x16": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "comp_gemm_f32_simt": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "comp_gemm_f32x16_variant": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "comp_gemm_f16x2": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "comp_gemm_f16x2_variant": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "comp_gemm_workspace_bytes": (_i64, [_i64, _i64]),
    "comp_gemm_workspace_bytes_mnk": (_i64, [_i64, _i64, _i64]),
    "comp_gemm_f32x16_ws": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp]),
    "comp_geglu_f32": (_int, [_vp, _vp, _vp, _i64, _vp]),
    "comp_gemm_f32x16_epilogue": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp]),
    "comp_gemm_f16x2_epilogue": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "comp_gemm_f32x16_noalloc": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "comp_device_status": (_int, [_vp, ctypes.POINTER(_u32)]),
    "comp_check_wait_timeout": (_int, [_vp]),
    "comp_check_stalled_pipeline": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "comp_status_string": (ctypes.c_char_p, [_int]),
    "comp_version": (_int, []),
}

_lock = threading.Lock()
_lib = None


class CompError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {status_string(status)}")


def load() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()'); there is no fallback"
            )
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().comp_status_string(int(status)).decode()


def call(name: str, *args) -> None:
    """Call an entry point that returns comp_status_t; raise CompError unless COMP_OK."""
    st = getattr(load(), name)(*args)
    if st != COMP_OK:
        raise CompError(st, name)


def device_status(stream: int | None = None) -> tuple[int, int]:
    """(status, fault word) after waiting for `stream`."""
    where = _u32(0)
    st = load().comp_device_status(stream, ctypes.byref(where))
    return int(st), int(where.value)
