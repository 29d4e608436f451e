"""The C ABI library on the host: it builds, loads, exports every symbol the
header declares, and rejects bad arguments before touching any device (these
calls never launch a kernel, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "compfp32.h")


@pytest.fixture(scope="session")
def lib():
    from compensated_fp32_projection_gb300 import _native, build

    build.build()
    return _native.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(comp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_calls():
    names = _declared()
    for n in ("comp_split_f32", "comp_merge_f32", "comp_gemm_f32x16", "comp_gemm_f32_simt", "comp_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from compensated_fp32_projection_gb300 import _native

    for name in _declared():
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, f"binding lacks {name}"


def test_status_strings_and_version(lib):
    for code in range(6):
        s = lib.comp_status_string(code).decode()
        assert s.startswith("COMP_")
    assert lib.comp_version() >= 100


P = ctypes.c_void_p


def test_split_argument_errors(lib):
    # negative size, NULL pointers, overlapping outputs: rejected before any device work
    assert lib.comp_split_f32(P(4096), P(1 << 20), P(1 << 21), -1, None) == 1
    assert lib.comp_split_f32(None, P(1 << 20), P(1 << 21), 8, None) == 1
    assert lib.comp_split_f32(P(4096), None, P(1 << 21), 8, None) == 1
    assert lib.comp_split_f32(P(4096), P(1 << 20), P(1 << 20) , 8, None) == 1  # hi == lo
    assert lib.comp_split_f32(P(4096), P(4096 + 8), P(1 << 21), 8, None) == 1  # hi inside x
    assert lib.comp_split_f32(P(4096), P(1 << 20), P((1 << 20) + 14), 8, None) == 1  # lo overlaps hi
    assert lib.comp_split_f32(None, None, None, 0, None) == 0  # empty is a no-op


def test_merge_argument_errors(lib):
    assert lib.comp_merge_f32(P(4096), P(1 << 20), P(1 << 21), -5, None) == 1
    assert lib.comp_merge_f32(None, P(1 << 20), P(1 << 21), 4, None) == 1
    assert lib.comp_merge_f32(P(4096), P(1 << 20), P(4096 + 4), 4, None) == 1  # partial overlap with acc_hi
    assert lib.comp_merge_f32(P(4096), P(1 << 20), P((1 << 20) - 4), 4, None) == 1  # partial overlap with acc_lo
    assert lib.comp_merge_f32(None, None, None, 0, None) == 0


def test_gemm_argument_errors(lib):
    for fn in (lib.comp_gemm_f32x16, lib.comp_gemm_f32_simt):
        assert fn(P(4096), P(1 << 20), P(1 << 24), -1, 4, 4, None) == 1
        assert fn(P(4096), P(1 << 20), P(1 << 24), 4, -1, 4, None) == 1
        assert fn(P(4096), P(1 << 20), P(1 << 24), 4, 4, -1, None) == 1
        assert fn(None, P(1 << 20), P(1 << 24), 4, 4, 4, None) == 1
        assert fn(P(4096), P(1 << 20), None, 4, 4, 4, None) == 1
        assert fn(P(4096), P(1 << 20), P(4096 + 16), 4, 4, 4, None) == 1  # y overlaps x
        assert fn(P(4096), P(1 << 20), P((1 << 20) + 4), 4, 4, 4, None) == 1  # y overlaps W
        assert fn(P(4096), P(1 << 20), P(1 << 24), 1 << 40, 1 << 40, 4, None) == 1  # M*N overflows
        assert fn(P(4096), P(1 << 20), P(1 << 24), 1 << 31, 4, 4, None) == 1  # M beyond int32
        assert fn(None, None, None, 0, 5, 7, None) == 0  # empty output: no-op
    assert lib.comp_gemm_f32x16_variant(P(4096), P(1 << 20), P(1 << 24), 4, 4, 4, 7, None) == 1
    # variant 3 (split fused into the swapped-operand kernel): M <= 32, K % 8 == 0, aligned x and W
    assert lib.comp_gemm_f32x16_variant(P(4096), P(1 << 20), P(1 << 24), 33, 4096, 64, 3, None) == 1
    assert lib.comp_gemm_f32x16_variant(P(4096), P(1 << 20), P(1 << 24), 16, 4096, 60, 3, None) == 1
    assert lib.comp_gemm_f32x16_variant(P(4096 + 4), P(1 << 20), P(1 << 24), 16, 4096, 64, 3, None) == 1
    assert lib.comp_gemm_f32x16_variant(P(4096), P((1 << 20) + 2), P(1 << 24), 16, 4096, 64, 3, None) == 1


def test_two_pass_argument_errors(lib):
    f2, ws = lib.comp_gemm_f16x2, lib.comp_gemm_f32x16_ws
    # comp_gemm_f16x2(hi, lo, W, y, M, N, K, stream)
    assert f2(P(4096), P(1 << 16), P(1 << 20), P(1 << 24), -1, 4, 8, None) == 1
    assert f2(None, P(1 << 16), P(1 << 20), P(1 << 24), 4, 4, 8, None) == 1
    assert f2(P(4096), P(1 << 16), P(1 << 20), P(4096 + 32), 4, 4, 8, None) == 1  # y overlaps hi
    assert f2(P(4096), P(1 << 16), P(1 << 20), P(1 << 24), 1 << 40, 1 << 40, 8, None) == 1
    assert f2(None, None, None, None, 0, 4, 8, None) == 0
    assert lib.comp_gemm_f16x2_variant(P(4096), P(1 << 16), P(1 << 20), P(1 << 24), 4, 4, 8, 4, None) == 1
    assert lib.comp_gemm_f16x2_variant(P(4096), P(1 << 16), P(1 << 20), P(1 << 24), 33, 4, 8, 3, None) == 1
    assert lib.comp_gemm_f16x2_variant(P(4096), P(1 << 16), P(1 << 20), P(1 << 24), 4, 4, 8, -1, None) == 1
    # comp_gemm_f32x16_ws(x, W, y, M, N, K, workspace, bytes, stream)
    assert ws(P(4096), P(1 << 20), P(1 << 24), -1, 4, 4, P(1 << 26), 64, None) == 1
    assert ws(None, None, None, 0, 4, 4, None, 0, None) == 0


def test_epilogue_argument_errors(lib):
    ep, e2 = lib.comp_gemm_f32x16_epilogue, lib.comp_gemm_f16x2_epilogue
    # comp_gemm_f32x16_epilogue(x, W, bias, gate, y, M, N, K, workspace, bytes, stream): 4 x 8 output at 1 << 24
    y = 1 << 24
    assert ep(P(4096), P(1 << 20), P(y + 4), None, P(y), 4, 8, 8, None, 0, None) == 1  # bias overlaps y
    assert ep(P(4096), P(1 << 20), None, P(y + 64), P(y), 4, 8, 8, None, 0, None) == 1  # gate overlaps y
    assert ep(P(4096), P(1 << 20), None, None, P(y), -1, 8, 8, None, 0, None) == 1
    assert ep(None, None, None, None, None, 0, 8, 8, None, 0, None) == 0  # empty output: no-op
    # comp_gemm_f16x2_epilogue(hi, lo, W, bias, gate, y, M, N, K, variant, stream)
    assert e2(P(4096), P(1 << 16), P(1 << 20), P(y + 28), None, P(y), 4, 8, 8, 0, None) == 1
    assert e2(P(4096), P(1 << 16), P(1 << 20), None, None, P(y), 4, 8, 8, 4, None) == 1  # variant out of range


def test_geglu_argument_errors(lib):
    f = lib.comp_geglu_f32
    # comp_geglu_f32(gate, up, out, n, stream)
    assert f(P(4096), P(1 << 16), P(1 << 20), -1, None) == 1
    assert f(None, P(1 << 16), P(1 << 20), 8, None) == 1
    assert f(P(4096), P(1 << 16), P(4096 + 4), 8, None) == 1  # out partly overlaps gate
    assert f(P(4096), P(1 << 16), P((1 << 16) + 4), 8, None) == 1  # out partly overlaps up
    assert f(None, None, None, 0, None) == 0  # n = 0: no-op


def test_workspace_bytes_mnk(lib):
    assert lib.comp_gemm_workspace_bytes_mnk(1000, 771, 1027) == 4 * 1000 * 1032 + 2 * 771 * 1032
    assert lib.comp_gemm_workspace_bytes_mnk(4096, 4096, 4096) == 4 * 4096 * 4096 + 2 * 4096 * 4096
    assert lib.comp_gemm_workspace_bytes_mnk(0, 0, 5) == 0
    assert lib.comp_gemm_workspace_bytes_mnk(-1, 4, 4) == 0
    assert lib.comp_gemm_workspace_bytes_mnk(1 << 40, 4, 1 << 30) == 0  # overflows


def test_workspace_bytes(lib):
    assert lib.comp_gemm_workspace_bytes(4096, 4096) == 4 * 4096 * 4096
    assert lib.comp_gemm_workspace_bytes(0, 77) == 0
    assert lib.comp_gemm_workspace_bytes(-1, 8) == 0
    assert lib.comp_gemm_workspace_bytes(1 << 40, 1 << 30) == 0  # overflows


def test_no_device_is_an_error_not_a_fallback(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments on a host without a usable sm_103 device: an error, never a CPU path
    assert lib.comp_split_f32(P(4096), P(1 << 20), P(1 << 21), 8, None) == 2
    assert lib.comp_gemm_f32x16(P(4096), P(1 << 20), P(1 << 24), 4, 4, 4, None) == 2
    assert lib.comp_gemm_f16x2(P(4096), P(1 << 16), P(1 << 20), P(1 << 24), 4, 4, 8, None) == 2
    assert lib.comp_gemm_f32x16_ws(P(4096), P(1 << 20), P(1 << 24), 4, 4, 4, P(1 << 26), 64, None) == 2


def test_package_import_does_not_need_the_library():
    import compensated_fp32_projection_gb300 as pkg

    assert callable(pkg.comp_gemm_f32x16)
