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
SOURCES = [os.path.join(CSRC, f) for f in ("ar.cu", "ar_kernels_f32.cu", "ar_kernels_f16.cu", "ar_kernels_bf16.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ar_kernels.cuh", "ar_kernels_ex.cuh", "ar_kernels_tma.cuh",
                                                   "ar_dispatch.h")] + [os.path.join(INCLUDE, "ar.h")]

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit in parallel, then link the shared
    library (written under a temporary name and renamed into place)."""
    if not force and not stale():
        return LIB
    with tempfile.TemporaryDirectory(dir=HERE, prefix="_build_") as tmpdir:
        objs, procs = [], []
        for src in SOURCES:
            obj = os.path.join(tmpdir, os.path.basename(src) + ".o")
            cmd = [NVCC, *ARCH, *FLAGS, "-c", "-o", obj, src]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append(subprocess.Popen(cmd))
            objs.append(obj)
        codes = [p.wait() for p in procs]
        if any(codes):
            raise RuntimeError(f"nvcc failed ({codes})")
        tmp = os.path.join(tmpdir, "libtps_ar.so")
        subprocess.run([NVCC, *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
