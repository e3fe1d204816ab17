"""ar_reduce_host_noalloc: the host entry point for callers that may not
allocate device memory (for instance a plug-in inside a framework whose
allocator owns the device memory, or a path that cannot afford
cudaMalloc's synchronisation).  It stages through the library's built-in
device area instead of caller-provided buffers.

Two calls in a row through the C ABI are compared bit for bit (any NaN
matches any NaN, as everywhere in this suite) with ar_reduce_host using
device staging buffers the test allocates; the second call also checks that
what the first call left in the shared area does not leak into the next.
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import tensor_partial_sum_gb300 as tps
from tensor_partial_sum_gb300 import workloads as W
from tests.libcasts import assert_same

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_partial_sum_gb300 import build
    build.build()
    yield
    tps.ar_free()


def reference(srcs, w, n_dsts):
    """The existing entry point, with device staging the test allocates."""
    h_srcs = [torch.from_numpy(s) for s in srcs]
    h_dsts = [torch.empty(w.nelem, dtype=torch.float32).pin_memory() for _ in range(n_dsts)]
    d_srcs = [torch.empty(w.nelem, device="cuda") for _ in srcs]
    d_dsts = [torch.empty(w.nelem, device="cuda") for _ in range(n_dsts)]
    tps.ar_reduce_host(h_srcs, h_dsts, d_srcs, d_dsts, nelem=w.nelem, dst_dtype="f32", wire_dtype=w.wire)
    torch.cuda.synchronize()
    return [h.numpy().copy() for h in h_dsts]


def test_two_calls_match_the_staged_entry_point():
    w = W.WORKLOADS["tp_small"]  # R=2 f32[32,4096], bf16 wire, 2 destinations: 2 MiB staged
    tps.ar_init(w.R, w.nelem)
    stream = torch.cuda.Stream()
    for call in range(2):
        srcs = [s * np.float32(1 + call) for s in W.generate(w)]  # different data on each call
        exp = reference(srcs, w, w.n_dsts)
        outs = [np.full(w.nelem, np.nan, dtype=np.float32) for _ in range(w.n_dsts)]  # pageable host memory
        tps.ar_reduce_host_noalloc(srcs, outs, nelem=w.nelem, dst_dtype="f32", wire_dtype=w.wire, stream=stream)
        stream.synchronize()
        for o, e in zip(outs, exp):
            assert_same(o, e, "f32", f"no-alloc call {call}")


def test_too_large_is_refused_and_writes_nothing():
    R, n_dsts = 2, 2
    per_buffer = tps.ar.AR_NOALLOC_SCRATCH_BYTES // (R + n_dsts) // 4  # f32 elements that just fit
    n = per_buffer + 1024
    tps.ar_init(R, n)
    srcs = [np.ones(n, dtype=np.float32) for _ in range(R)]
    outs = [np.full(n, 7.0, dtype=np.float32) for _ in range(n_dsts)]
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce_host_noalloc(srcs, outs, nelem=n, dst_dtype="f32", wire_dtype="bf16")
    assert e.value.status == 3
    assert all((o == 7.0).all() for o in outs)
    # the largest call that fits works and matches the arithmetic (1 + 1 = 2)
    tps.ar_reduce_host_noalloc(srcs, outs, nelem=per_buffer, dst_dtype="f32", wire_dtype="bf16")
    torch.cuda.synchronize()
    assert all((o[:per_buffer] == 2.0).all() and (o[per_buffer:] == 7.0).all() for o in outs)
