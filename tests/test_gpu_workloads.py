"""GPU parity at full workload sizes, in the launch configuration the
benchmark uses: automatic variant choice, a CUDA graph on a created stream,
launches back to back as programmatic dependents.

Every element of every destination is compared with the oracle, bit for bit
(any NaN matches any NaN).  The oracle runs over contiguous ranges on every
host core (tests/whole.py), which takes about a second for the largest
workload."""
import numpy as np
import pytest
import torch

import oracle
import tensor_partial_sum_gb300 as tps
from tensor_partial_sum_gb300 import workloads as W
from tests import whole
from tests.gpu_util import TORCH_DTYPE, to_device, to_host
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


def as_benchmarked(call, outs):
    """Run ``call(stream)`` the way the benchmark times it: inside a CUDA
    graph on a created stream, two launches back to back (so the second is a
    programmatic dependent of the first), replayed after the outputs were
    poisoned."""
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        call(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
        call(s)
    for o in outs:
        o.view(torch.uint8).fill_(0x7F)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    del g


@pytest.mark.parametrize("name", ["tp_small", "prefill", "bf16_t3", "f16_edges"])
def test_full_size_workload(name):
    w = W.WORKLOADS[name]
    srcs = W.generate(w)
    tps.ar_init(w.R, w.nelem)
    src_t = [to_device(s, w.dst) for s in srcs]
    dst_t = [torch.empty(w.nelem, dtype=TORCH_DTYPE[w.dst], device="cuda") for _ in range(w.n_dsts)]
    as_benchmarked(lambda s: tps.ar_reduce(src_t, dst_t, nelem=w.nelem, dst_dtype=w.dst, wire_dtype=w.wire,
                                           stream=s), dst_t)
    del src_t
    exp = whole.reduce(srcs, w.dst, w.wire)
    for d, t in enumerate(dst_t):
        assert_same(to_host(t, w.dst), exp, w.dst, f"{name} destination {d}, all {w.nelem} elements")


@pytest.mark.parametrize("dst,wire", [(d, w) for d in ("f32", "f16", "bf16") for w in ("f32", "f16", "bf16")])
def test_every_dtype_pair_at_prefill_size(dst, wire):
    """Every (T_dst, T_wire) pair at the prefill shape (R=2 [2048,4096], 2
    destinations) on edge-laden inputs (normals, f16-overflowing values,
    subnormals, signed zeros, infinities, NaN, ties), launched as the
    benchmark launches; every element compared with the oracle."""
    from tests.libcasts import lib_round
    from tests.test_oracle_fold import edgy_f32
    n = 2048 * 4096
    rng = np.random.Generator(np.random.PCG64(4096 + len(dst) * 7 + len(wire)))
    srcs = [lib_round(dst, edgy_f32(rng, n)) for _ in range(2)]
    tps.ar_init(2, n)
    src_t = [to_device(a, dst) for a in srcs]
    dst_t = [torch.empty(n, dtype=TORCH_DTYPE[dst], device="cuda") for _ in range(2)]
    as_benchmarked(lambda s: tps.ar_reduce(src_t, dst_t, nelem=n, dst_dtype=dst, wire_dtype=wire, stream=s), dst_t)
    exp = whole.reduce(srcs, dst, wire)
    for d, t in enumerate(dst_t):
        assert_same(to_host(t, dst), exp, dst, f"{dst}/{wire} destination {d}, all {n} elements")


def test_decode_every_call_graph_captured():
    """The decode workload exactly as benchmarked: 10000 calls with their own
    buffers captured in one CUDA graph; every output element of every call is
    compared with the oracle."""
    w = W.WORKLOADS["decode"]
    row = (w.nelem + 3) // 4 * 4
    buf = torch.zeros((w.calls, w.R + w.n_dsts, row), dtype=torch.float32, device="cuda")
    host = np.zeros((w.calls, w.R, w.nelem), dtype=np.float32)
    for k in range(w.calls):
        host[k] = np.stack(W.generate(w, call=k))
    buf[:, :w.R, :w.nelem].copy_(torch.from_numpy(host))
    tps.ar_init(w.R, w.nelem)
    p0, sc, sb = buf.data_ptr(), buf.stride(0) * 4, buf.stride(1) * 4
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for k in range(w.calls):
            tps.ar_reduce([p0 + k * sc + r * sb for r in range(w.R)],
                          [p0 + k * sc + (w.R + d) * sb for d in range(w.n_dsts)],
                          nelem=w.nelem, dst_dtype="f32", wire_dtype=w.wire, stream=stream)
    g.replay()
    torch.cuda.synchronize()
    assert tps.ar_query("last_variant") == tps.ar.VARIANTS["latency"]
    out = buf[:, w.R:, :w.nelem].cpu().numpy()
    flat = [host[:, r, :].ravel() for r in range(w.R)]
    exp = oracle.reduce(flat, 1, "f32", w.wire)[0].reshape(w.calls, w.nelem)
    for d in range(w.n_dsts):
        assert_same(out[:, d, :].ravel(), exp.ravel(), "f32", f"decode destination {d}")


@pytest.mark.parametrize("name", ["prefill_residual", "prefill_bias", "prefill_strided", "prefill_inactive",
                                  "prefill_pack"])
def test_full_size_extended_workload(name):
    """The extended entry points at the prefill size, set up as the benchmark
    sets them up; every row of every destination is compared with the
    oracle, and the row padding must stay untouched."""
    w = W.WORKLOADS[name]
    srcs = W.generate(w)
    ne0, ne1, pad, es = w.ne0, w.ne1, w.row_pad, w.elem_bytes
    tdt = TORCH_DTYPE[w.dst]
    tps.ar_init(w.R, w.nelem)

    def rows_tensor(a=None):
        t = torch.zeros((ne1, ne0 + pad), dtype=tdt, device="cuda")
        if a is not None:
            t[:, :ne0].copy_(to_device(a, w.dst).view(ne1, ne0))
        return t

    if w.op == "pack":
        src = to_device(srcs[0], w.dst)
        out = torch.empty(w.nelem, dtype=TORCH_DTYPE[w.wire], device="cuda")
        as_benchmarked(lambda s: tps.ar_wire_pack(src, out, dst_dtype=w.dst, wire_dtype=w.wire, stream=s), [out])
        assert_same(to_host(out, w.wire), whole.wire_pack(srcs[0], w.dst, w.wire), w.wire, name)
        return
    s_t = [None if r in w.inactive else rows_tensor(srcs[r]) for r in range(w.R)]
    d_t = [rows_tensor() for _ in range(w.n_dsts)]
    res_t = to_device(srcs[w.R], w.dst) if w.residual else None
    layout = tps.make_layout(ne0, ne1, src_row_bytes=[(ne0 + pad) * es] * w.R,
                             dst_row_bytes=[(ne0 + pad) * es] * w.n_dsts, residual=res_t,
                             residual_row_bytes=0 if w.residual == "row" else None, inactive=w.inactive)
    as_benchmarked(lambda s: tps.ar_reduce_ex(s_t, d_t, layout, w.dst, w.wire, stream=s),
                   [d[:, :ne0] for d in d_t])
    exp = whole.reduce_rows(srcs[:w.R], w.dst, w.wire, ne0, ne1, inactive=w.inactive,
                            residual=srcs[w.R] if w.residual else None, residual_kind=w.residual)
    for k, d in enumerate(d_t):
        got = to_host(d[:, :ne0].contiguous(), w.dst)
        assert_same(got, exp, w.dst, f"{name} destination {k}, all rows")
        if pad:
            assert (d[:, ne0:] == 0).all(), "row padding written"
