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


STATUS_VALUES = {
    # the numbering of the boundary's status enum; part of the ABI
    "COMP_OK": 0,
    "COMP_ERR_INVALID_VALUE": 1,
    "COMP_ERR_MISALIGNED": 2,
    "COMP_ERR_UNSUPPORTED_DEVICE": 3,
    "COMP_ERR_LAUNCH": 4,
    "COMP_ERR_TIMEOUT": 5,
    "COMP_ERR_CUDA": 6,
}


def test_status_values_pinned():
    """Every code's numeric value in the header, and the binding's copy of it."""
    from compensated_fp32_projection_gb300 import _native

    text = open(HEADER).read()
    body = re.search(r"typedef enum comp_status \{(.*?)\} comp_status_t;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    found = {k: int(v) for k, v in re.findall(r"(COMP_[A-Z_]+)\s*=\s*(\d+)", body)}
    assert found == STATUS_VALUES
    for name, value in STATUS_VALUES.items():
        assert getattr(_native, name) == value, name


def test_status_strings_and_version(lib):
    for name, code in STATUS_VALUES.items():
        s = lib.comp_status_string(code).decode()
        assert s.split(":")[0] == name
    assert lib.comp_status_string(99).decode() == "unknown comp_status_t"
    assert lib.comp_version() >= 100


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "compfp32.h"

static int check(comp_status_t s, int value, const char* name)
{
    const char* str = comp_status_string(s);
    if ((int)s != value || strncmp(str, name, strlen(name)) != 0) {
        printf("bad %s\n", name);
        return 1;
    }
    return 0;
}

int main(void)
{
    int bad = 0;
    bad += check(COMP_OK, 0, "COMP_OK");
    bad += check(COMP_ERR_INVALID_VALUE, 1, "COMP_ERR_INVALID_VALUE");
    bad += check(COMP_ERR_MISALIGNED, 2, "COMP_ERR_MISALIGNED");
    bad += check(COMP_ERR_UNSUPPORTED_DEVICE, 3, "COMP_ERR_UNSUPPORTED_DEVICE");
    bad += check(COMP_ERR_LAUNCH, 4, "COMP_ERR_LAUNCH");
    bad += check(COMP_ERR_TIMEOUT, 5, "COMP_ERR_TIMEOUT");
    bad += check(COMP_ERR_CUDA, 6, "COMP_ERR_CUDA");
    /* argument errors need no device: a negative size is rejected first */
    if (comp_split_f32((const float*)0, (uint16_t*)0, (uint16_t*)0, -1, (comp_stream_t)0) != COMP_ERR_INVALID_VALUE)
        ++bad;
    if (comp_gemm_workspace_bytes(4096, 4096) != 4LL * 4096 * 4096)
        ++bad;
    printf(bad ? "FAIL\n" : "OK\n");
    return bad;
}
"""


def test_header_compiles_as_c11_and_links(lib, tmp_path):
    """A plain C11 program includes the header, links the library and reads
    every status code's value and name through it."""
    import shutil
    import subprocess

    from compensated_fp32_projection_gb300 import _native

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(_native.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-l:libcompfp32.so", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "OK", out.stdout + out.stderr


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
    assert lib.comp_gemm_f16x2_variant(P(4096), P(1 << 16), P(1 << 20), P(1 << 24), 4, 4, 8, 5, None) == 1
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
    assert e2(P(4096), P(1 << 16), P(1 << 20), None, None, P(y), 4, 8, 8, 5, None) == 1  # variant out of range


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
    unsupported = STATUS_VALUES["COMP_ERR_UNSUPPORTED_DEVICE"]
    assert lib.comp_split_f32(P(4096), P(1 << 20), P(1 << 21), 8, None) == unsupported
    assert lib.comp_gemm_f32x16(P(4096), P(1 << 20), P(1 << 24), 4, 4, 4, None) == unsupported
    assert lib.comp_gemm_f16x2(P(4096), P(1 << 16), P(1 << 20), P(1 << 24), 4, 4, 8, None) == unsupported
    assert lib.comp_gemm_f32x16_ws(P(4096), P(1 << 20), P(1 << 24), 4, 4, 4, P(1 << 26), 64, None) == unsupported


def test_package_import_does_not_need_the_library():
    import compensated_fp32_projection_gb300 as pkg

    assert callable(pkg.comp_gemm_f32x16)
