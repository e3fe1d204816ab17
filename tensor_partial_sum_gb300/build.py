"""Compile the CUDA library in-tree for sm_103a.

``python -m tensor_partial_sum_gb300.build`` (or ``build()``) writes
``libtps_ar.so`` next to this file.  nvcc cross-compiles, so this also runs
on a machine without a GPU.  The host code is portable C++ (x86_64 and
aarch64 build the same sources).
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libtps_ar.so")
SOURCES = [os.path.join(CSRC, "ar.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ar_kernels.cuh"), os.path.join(INCLUDE, "ar.h")]

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
         "-I" + INCLUDE, "-I" + CSRC]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
    os.close(fd)
    cmd = [NVCC, *ARCH, *FLAGS, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    try:
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
