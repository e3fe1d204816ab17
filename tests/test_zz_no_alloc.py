"""ar_reduce_host_noalloc: the host entry point for callers that may not
allocate device memory (for instance a plug-in inside a framework whose
allocator owns the device memory, or a path that cannot afford
cudaMalloc's synchronisation).  It stages through the library's built-in
device area instead of caller-provided buffers.

Two calls in a row through the C ABI are compared bit for bit (any NaN
matches any NaN, as everywhere in this suite) with the oracle and with
ar_reduce_host using device staging buffers the test allocates; the second
call also checks that what the first call left in the shared area does not
leak into the next.  This file is collected last on purpose."""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import tensor_partial_sum_gb300 as tps
from tensor_partial_sum_gb300 import workloads as W
from tests.libcasts import assert_same

pytestmark = pytest.mark.gpu

OVERLAP, TOO_LARGE = 5, 3


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_partial_sum_gb300 import build
    build.build()
    yield
    tps.ar_free()


def staged(srcs, w, n_dsts):
    """The existing entry point, with device staging the test allocates."""
    h_srcs = [torch.from_numpy(s) for s in srcs]
    h_dsts = [torch.empty(w.nelem, dtype=torch.float32).pin_memory() for _ in range(n_dsts)]
    d_srcs = [torch.empty(w.nelem, device="cuda") for _ in srcs]
    d_dsts = [torch.empty(w.nelem, device="cuda") for _ in range(n_dsts)]
    tps.ar_reduce_host(h_srcs, h_dsts, d_srcs, d_dsts, nelem=w.nelem, dst_dtype="f32", wire_dtype=w.wire)
    torch.cuda.synchronize()
    return [h.numpy().copy() for h in h_dsts]


def test_two_calls_match_the_oracle_and_the_staged_entry_point():
    w = W.WORKLOADS["tp_small"]  # R=2 f32[32,4096], bf16 wire, 2 destinations: 2 MiB staged
    tps.ar_init(w.R, w.nelem)
    stream = torch.cuda.Stream()
    for call in range(2):
        srcs = [s * np.float32(1 + call) for s in W.generate(w)]  # different data on each call
        exp = oracle.reduce(srcs, 1, w.dst, w.wire)[0]
        via_staging = staged(srcs, w, w.n_dsts)
        outs = [np.full(w.nelem, np.nan, dtype=np.float32) for _ in range(w.n_dsts)]  # pageable host memory
        tps.ar_reduce_host_noalloc(srcs, outs, nelem=w.nelem, dst_dtype="f32", wire_dtype=w.wire, stream=stream)
        stream.synchronize()
        for d, (o, v) in enumerate(zip(outs, via_staging)):
            assert_same(o, exp, "f32", f"no-alloc call {call} destination {d} against the oracle")
            assert_same(o, v, "f32", f"no-alloc call {call} destination {d} against ar_reduce_host")


def test_too_large_is_refused_and_the_largest_fitting_call_works():
    R, n_dsts = 2, 2
    per_buffer = tps.ar.AR_NOALLOC_SCRATCH_BYTES // (R + n_dsts) // 4  # f32 elements that just fit
    n = per_buffer + 1024
    tps.ar_init(R, n)
    srcs = W.generate("prefill", nelem=n)[:R]  # the prefill recipe: N(0,1) with 0.1% outliers x50
    outs = [np.full(n, 7.0, dtype=np.float32) for _ in range(n_dsts)]
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce_host_noalloc(srcs, outs, nelem=n, dst_dtype="f32", wire_dtype="bf16")
    assert e.value.status == TOO_LARGE
    assert all((o == 7.0).all() for o in outs)
    tps.ar_reduce_host_noalloc(srcs, outs, nelem=per_buffer, dst_dtype="f32", wire_dtype="bf16")
    torch.cuda.synchronize()
    exp = oracle.reduce([s[:per_buffer] for s in srcs], 1, "f32", "bf16")[0]
    for o in outs:
        assert_same(o[:per_buffer], exp, "f32", "largest no-alloc call")
        assert (o[per_buffer:] == 7.0).all()


def test_partly_overlapping_host_buffers_are_refused():
    """A host destination that partly overlaps a host source would be
    overwritten while the copies in still read it: refused before anything
    is enqueued.  A destination that is exactly a source stays allowed."""
    R, n = 2, 100_000
    tps.ar_init(R, n)
    back = W.generate("prefill", nelem=3 * n)[0]
    before = back.copy()
    srcs = [back[:n], back[2 * n:]]
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce_host_noalloc(srcs, [back[n // 2:n // 2 + n]], nelem=n, dst_dtype="f32", wire_dtype="bf16")
    assert e.value.status == OVERLAP
    other = np.zeros(2 * n, dtype=np.float32)
    with pytest.raises(tps.ARError) as e:  # two destinations that share bytes
        tps.ar_reduce_host_noalloc(srcs, [other[:n], other[n // 4:n // 4 + n]], nelem=n, dst_dtype="f32",
                                   wire_dtype="bf16")
    assert e.value.status == OVERLAP
    torch.cuda.synchronize()
    assert np.array_equal(back.view(np.uint32), before.view(np.uint32)) and not other.any()
    exp = oracle.reduce([s.copy() for s in srcs], 1, "f32", "bf16")[0]
    tps.ar_reduce_host_noalloc(srcs, [srcs[1]], nelem=n, dst_dtype="f32", wire_dtype="bf16")
    torch.cuda.synchronize()
    assert_same(back[2 * n:], exp, "f32", "no-alloc in place")


def test_a_device_reset_between_contexts(tmp_path):
    """A plain C program: a call, ar_free, cudaDeviceReset, ar_init, another
    call (in a process of its own, so the reset ends only that process's
    context).  The second call must use the staging area's address in the
    new context, not the one the first call looked up."""
    from tests.test_c_abi import CUDA, _compile
    exe = _compile("noalloc_reset.c", str(tmp_path / "noalloc_reset"), cflags=["-I", os.path.join(CUDA, "include")],
                   ldflags=["-L", os.path.join(CUDA, "lib64"), "-lcudart",
                            f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout + out.stderr
