"""Builds the CUDA library ``libcompfp32.so`` in place (nvcc, sm_103a only).

Each ``csrc/*.cu`` is compiled in parallel to an object under ``_build/`` and
the objects are linked into one shared library next to this file.  The CUDA
runtime is linked statically, so the library needs only the NVIDIA driver at
run time (and loads, without running anything, on a machine with no GPU).

No fast-math and no flush-to-zero: the split and merge must be bit-exact.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libcompfp32.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3",
    "-lineinfo",
    "-std=c++17",
    "-Xcompiler",
    "-fPIC",
    "-Xptxas",
    "-v",
    "-I",
    INCLUDE,
    "-I",
    CSRC,
]


def nvcc() -> str:
    env = os.environ.get("NVCC")
    if env:
        return env
    found = shutil.which("nvcc")
    if found:
        return found
    return "/usr/local/cuda/bin/nvcc"


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return _sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)
    ] + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, "-c", src, "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
    return obj, p.stderr


# Kernels that move registers between warpgroups with setmaxnreg assume this
# launch register count; a different count could make setmaxnreg.inc wait
# forever, so the build refuses it.
SETMAXNREG_KERNELS = {"comp_gemm_kernel": 96, "comp_f16x2_kernel": 168, "comp_f16x2_pair_kernel": 168,
                      "comp_f16x2_splitk_kernel": 168, "comp_f32x16_pair_kernel": 128}


def _check_register_budget(ptxas_log: str) -> None:
    current = None
    for line in ptxas_log.splitlines():
        if "Compiling entry function" in line:
            current = next((k for k in SETMAXNREG_KERNELS if k in line), None)
        elif current and "Used" in line and "registers" in line:
            used = int(line.split("Used")[1].split("registers")[0])
            if used != SETMAXNREG_KERNELS[current]:
                raise RuntimeError(f"{current}: ptxas reports {used} registers, the register split assumes "
                                   f"{SETMAXNREG_KERNELS[current]}")
            current = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if any source changed; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(_compile, srcs))
    with open(os.path.join(BUILD, "ptxas.txt"), "w") as f:
        for (obj, log), src in zip(results, srcs):
            f.write(f"== {os.path.basename(src)}\n{log}\n")
    _check_register_budget("\n".join(log for _, log in results))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(open(os.path.join(BUILD, "ptxas.txt")).read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
