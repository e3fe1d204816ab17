"""The C ABI used from plain C: include/ar.h compiles as C11 with gcc on its
own, links against libtps_ar.so, and (on a GPU) a C program reduces
cudaMalloc'd buffers through ar_init / ar_reduce / ar_free."""
import os
import shutil
import subprocess

import pytest
import torch

from tensor_partial_sum_gb300 import build as B

HERE = os.path.dirname(os.path.abspath(__file__))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(src, out, cflags=(), ldflags=()):
    B.build()
    libdir = os.path.dirname(B.LIB)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", B.INCLUDE, *cflags,
           os.path.join(HERE, "c", src), "-o", out, "-L", libdir, "-ltps_ar", f"-Wl,-rpath,{libdir}", *ldflags]
    subprocess.run(cmd, check=True)
    return out


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_c11_and_host_calls_work(tmp_path):
    exe = _compile("abi_host.c", str(tmp_path / "abi_host"))
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_layout_struct_matches_the_binding(tmp_path):
    """ar_layout as a C compiler lays it out from the header has the size and
    field offsets of the binding's ctypes mirror (ArLayout)."""
    import ctypes
    from tensor_partial_sum_gb300 import ar as A
    exe = _compile("layout_offsets.c", str(tmp_path / "layout_offsets"))
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    c = {k: int(v) for k, v in (line.split() for line in out.stdout.splitlines())}
    assert c.pop("size") == ctypes.sizeof(A.ArLayout)
    assert c == {name: getattr(A.ArLayout, name).offset for name, _ in A.ArLayout._fields_}


@pytest.mark.gpu
def test_c_program_reduces_on_the_gpu(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile("abi_gpu.c", str(tmp_path / "abi_gpu"), cflags=["-I", os.path.join(CUDA, "include")],
                   ldflags=["-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout + out.stderr


@pytest.mark.gpu
def test_host_cost_of_a_decode_call(tmp_path):
    """Validating, choosing and enqueuing a decode-sized call from C costs
    a few microseconds at most (the figures are printed for the record)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile("host_cost.c", str(tmp_path / "host_cost"), cflags=["-I", os.path.join(CUDA, "include")],
                   ldflags=["-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout + out.stderr
    fields = dict(kv.split("=") for kv in out.stdout.split()[1:])
    print(out.stdout.strip())
    assert float(fields["eager_us"]) < 20 and float(fields["capture_us"]) < 20
