"""GPU parity: the CUDA path through the C ABI against the oracle, element
by element, bit for bit (any NaN matches any NaN).

Sizes are small enough for the oracle to finish in seconds yet span many
16-byte vectors, several CTA tiles and a ragged tail."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import tensor_partial_sum_gb300 as tps
from tensor_partial_sum_gb300 import workloads as W
from tests import whole
from tests.gpu_util import Ctx, check_guards, run, to_device, to_host
from tests.libcasts import assert_same, lib_round
from tests.test_oracle_fold import edgy_f32

pytestmark = pytest.mark.gpu

TYPES = ["f32", "f16", "bf16"]
PAIRS = list(itertools.product(TYPES, TYPES))
VARIANTS = ["auto", "latency", "bandwidth", "scalar", "naive", "tma"]


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_partial_sum_gb300 import build
    build.build()
    c = Ctx()
    yield c
    tps.ar_free()


def srcs_for(seed, R, n, dst):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [lib_round(dst, edgy_f32(rng, n)) for _ in range(R)]


def expect(srcs, dst, wire):
    return oracle.reduce(srcs, 1, dst, wire)[0]


@pytest.mark.parametrize("dst,wire", PAIRS)
@pytest.mark.parametrize("R", [1, 2, 3, 5, 8, 16])
def test_all_pairs_all_variants(ctx, dst, wire, R):
    n = 70001  # 17500 f32 vectors or 8750 16-bit vectors, plus a 1-element tail
    srcs = srcs_for(R * 31 + len(dst), R, n, dst)
    exp = expect(srcs, dst, wire)
    n_dsts = R % 4 + 1
    for v in VARIANTS:
        outs, backs = run(ctx, srcs, n_dsts, dst, wire, variant=v, pad=256)
        for d, o in enumerate(outs):
            assert_same(o, exp, dst, f"{dst}/{wire} R={R} variant={v} dst={d}")
        check_guards(backs)


SIZES = [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 33, 127, 128, 129, 255, 257, 1023, 1025,
         4095, 4096, 4097, 4099, 256 * 4 * 4 - 1, 256 * 4 * 4 + 3, 1_000_003]


@pytest.mark.parametrize("dst,wire", [("f32", "bf16"), ("bf16", "bf16"), ("f16", "f32")])
@pytest.mark.parametrize("n", SIZES)
def test_sizes_and_tails(ctx, dst, wire, n):
    srcs = srcs_for(n, 4, n, dst)
    exp = expect(srcs, dst, wire)
    for v in VARIANTS:
        outs, backs = run(ctx, srcs, 2, dst, wire, variant=v, pad=64)
        for o in outs:
            assert_same(o, exp, dst, f"n={n} variant={v}")
        check_guards(backs)


@pytest.mark.parametrize("variant", ["bandwidth", "scalar", "naive"])
@pytest.mark.parametrize("grid", [1, 2, 3, 7, 152, 1000])
def test_grid_size_does_not_change_bits(ctx, variant, grid):
    n = 300_007
    srcs = srcs_for(grid, 3, n, "f32")
    exp = expect(srcs, "f32", "f16")
    outs, _ = run(ctx, srcs, 1, "f32", "f16", variant=variant, grid=grid)
    assert_same(outs[0], exp, "f32", f"{variant} grid={grid}")


@pytest.mark.parametrize("dst", TYPES)
def test_unaligned_pointers(ctx, dst):
    """Buffers one element off 16-byte alignment take the element-wise path
    and give the same bits; a forced vector variant is refused."""
    n = 10_001
    srcs = srcs_for(5, 3, n, dst)
    exp = expect(srcs, dst, "bf16")
    outs, backs = run(ctx, srcs, 2, dst, "bf16", src_offsets=[1, 0, 3], dst_offsets=[0, 1], pad=64)
    for o in outs:
        assert_same(o, exp, dst, "unaligned")
    check_guards(backs)
    assert tps.ar_query("last_variant") == tps.ar.VARIANTS["scalar"]
    with pytest.raises(tps.ARError) as e:
        run(ctx, srcs, 1, dst, "bf16", variant="bandwidth", src_offsets=[1, 0, 0])
    assert e.value.status == 1


@pytest.mark.parametrize("dst,wire", PAIRS)
@pytest.mark.parametrize("R", [1, 2, 3, 5, 8, 16])
def test_mixed_offsets_every_pair(ctx, dst, wire, R):
    """Every source and destination at its own offset from a 16-byte
    boundary (any offset a 16-byte vector allows, destination 0 included),
    sizes from one element to a million with every kind of tail: AUTO's
    element-wise kernel gives the oracle's bits and leaves the poisoned
    margins around every destination alone."""
    V = 16 // (4 if dst == "f32" else 2)
    rng = np.random.Generator(np.random.PCG64(R * 97 + len(dst) + 3 * len(wire)))
    for n in (1, V - 1, V + 1, 3 * V + 2, 70_001, 1_000_003):
        srcs = srcs_for(n + R, R, n, dst)
        exp = expect(srcs, dst, wire)
        n_dsts = R % 3 + 1
        src_off = [int(x) for x in rng.integers(0, V, R)]
        dst_off = [int(x) for x in rng.integers(0, V, n_dsts)]
        if len(set(src_off + dst_off)) == 1:  # make sure the offsets differ
            dst_off[-1] = (dst_off[-1] + 1) % V
        outs, backs = run(ctx, srcs, n_dsts, dst, wire, src_offsets=src_off, dst_offsets=dst_off, pad=64)
        for d, o in enumerate(outs):
            assert_same(o, exp, dst, f"{dst}/{wire} R={R} n={n} offsets {src_off} -> {dst_off} dst={d}")
        check_guards(backs)
        assert tps.ar_query("last_variant") == tps.ar.VARIANTS["scalar"]


@pytest.mark.parametrize("dst", TYPES)
@pytest.mark.parametrize("off", [1, 2, 3, 4, 5, 7])
@pytest.mark.parametrize("variant", ["auto", "latency", "bandwidth"])
@pytest.mark.parametrize("n", [1, 2, 7, 9, 10_001, 300_007])
def test_common_offset_takes_the_vector_path(ctx, dst, off, variant, n):
    """Buffers that all sit the same number of elements off a vector
    boundary run the vector kernel on the aligned part, with the elements
    before it done one by one: same bits, margins intact, no fall-back to
    the element-wise kernel."""
    R = 3
    srcs = srcs_for(100 + off + n, R, n, dst)
    exp = expect(srcs, dst, "bf16")
    outs, backs = run(ctx, srcs, 2, dst, "bf16", variant=variant, src_offsets=[off] * R,
                      dst_offsets=[off, off], pad=64)
    for o in outs:
        assert_same(o, exp, dst, f"common offset {off}")
    check_guards(backs)
    want = "latency" if variant == "auto" else variant
    assert tps.ar_query("last_variant") == tps.ar.VARIANTS[want]


@pytest.mark.parametrize("variant", ["latency", "bandwidth"])
def test_common_offset_many_ranks_in_place(ctx, variant):
    """R = 16 with a shared odd offset, destination 0 one of the sources."""
    n, R = 123_457, 16
    srcs = srcs_for(77, R, n, "f32")
    exp = expect(srcs, "f32", "f16")
    outs, _ = run(ctx, srcs, 2, "f32", "f16", variant=variant, src_offsets=[3] * R,
                  dst_offsets=[3, 3], in_place=5)
    for o in outs:
        assert_same(o, exp, "f32", "R=16 offset 3 in place")
    assert tps.ar_query("last_variant") == tps.ar.VARIANTS[variant]


@pytest.mark.parametrize("grid", [1, 3, 152])
def test_common_offset_with_a_persistent_grid(ctx, grid):
    """The head is done by CTA 0 after its share of the rounds, whatever the
    grid; with a tail too, the last CTA does both jobs' elements."""
    n = 300_007
    srcs = srcs_for(300 + grid, 2, n, "bf16")
    exp = expect(srcs, "bf16", "f16")
    outs, backs = run(ctx, srcs, 2, "bf16", "f16", variant="bandwidth", grid=grid, src_offsets=[3, 3],
                      dst_offsets=[3, 3], pad=64)
    for o in outs:
        assert_same(o, exp, "bf16", f"offset 3, grid {grid}")
    check_guards(backs)


def test_tma_refuses_an_offset(ctx):
    """The bulk-copy variant needs 16-byte starts even when the offset is shared."""
    srcs = srcs_for(78, 2, 4096, "f32")
    with pytest.raises(tps.ARError) as e:
        run(ctx, srcs, 1, "f32", "bf16", variant="tma", src_offsets=[1, 1], dst_offsets=[1])
    assert e.value.status == 1


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("k", [0, 2])
def test_in_place(ctx, variant, k):
    """A destination may be one of the sources (the pages reduce in place)."""
    n = 50_003
    srcs = srcs_for(7 + k, 3, n, "f32")
    exp = expect(srcs, "f32", "bf16")
    outs, _ = run(ctx, srcs, 2, "f32", "bf16", variant=variant, in_place=k)
    for o in outs:
        assert_same(o, exp, "f32", f"in place into source {k}")


def test_auto_dispatch_by_size(ctx):
    ctx.ensure(4, 1 << 22)
    limit = tps.ar_query("latency_max_bytes")
    small = max(1, limit // (8 * 4) - 64)
    big = limit // (8 * 4) + 64
    for n, want in ((small, "latency"), (big, "bandwidth")):
        srcs = srcs_for(n, 4, n, "f32")
        outs, _ = run(ctx, srcs, 4, "f32", "f16")
        assert tps.ar_query("last_variant") == tps.ar.VARIANTS[want]
        assert_same(outs[0], expect(srcs, "f32", "f16"), "f32", f"auto n={n}")


def test_threshold_option_moves_dispatch(ctx):
    ctx.ensure(2, 1 << 20)
    old = tps.ar_query("latency_max_bytes")
    try:
        tps.ar_set_option("latency_max_bytes", 0)
        srcs = srcs_for(1, 2, 1000, "f32")
        run(ctx, srcs, 1, "f32", "bf16")
        assert tps.ar_query("last_variant") == tps.ar.VARIANTS["bandwidth"]
        tps.ar_set_option("latency_max_bytes", 1 << 40)
        run(ctx, srcs, 1, "f32", "bf16")
        assert tps.ar_query("last_variant") == tps.ar.VARIANTS["latency"]
    finally:
        tps.ar_set_option("latency_max_bytes", old)


def test_zero_elements_is_a_no_op(ctx):
    ctx.ensure(2, 1 << 16)
    d = torch.full((8,), 3.0, device="cuda")
    tps.ar_reduce([d, d], [d], nelem=0, dst_dtype="f32", wire_dtype="bf16")
    torch.cuda.synchronize()
    assert (d == 3.0).all()


def test_errors_write_nothing(ctx):
    tps.ar_init(2, 1000)
    ctx.R = None  # the next test re-initialises with its own limits
    a = torch.randn(1001, device="cuda")  # one element more than max_elems
    b = torch.randn(1001, device="cuda")
    out = torch.full((1001,), 7.0, device="cuda")
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce([a, b], [out], nelem=1001, dst_dtype="f32")
    assert e.value.status == 3
    with pytest.raises(ValueError):  # the binding: a destination shorter than the call
        tps.ar_reduce([a, b], [out[:500]], nelem=1000, dst_dtype="f32")
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce([a, b], [a[10:]], nelem=990, dst_dtype="f32")
    assert e.value.status == 5
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce([a], [out], nelem=1000, dst_dtype="f32")  # one source short of R=2
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert (out == 7.0).all()


def test_fault_injection_returns_status_and_writes_nothing(ctx):
    ctx.ensure(2, 1 << 16)
    a = torch.randn(4096, device="cuda")
    out = torch.full((4096,), 7.0, device="cuda")
    tps.ar_set_option("fault_inject", 1)
    try:
        with pytest.raises(tps.ARError) as e:
            tps.ar_reduce([a, a], [out], dst_dtype="f32")
        assert e.value.status == 6
    finally:
        tps.ar_set_option("fault_inject", 0)
    torch.cuda.synchronize()
    assert (out == 7.0).all()
    tps.ar_reduce([a, a], [out], dst_dtype="f32")  # and the context still works
    torch.cuda.synchronize()
    assert torch.equal(out, (a.to(torch.bfloat16).float() * 2))


def test_cuda_graph_capture_and_replay(ctx):
    ctx.ensure(4, 1 << 16)
    n = 4099
    srcs = srcs_for(11, 4, n, "f32")
    exp = expect(srcs, "f32", "f16")
    src_t = [to_device(s, "f32") for s in srcs]
    outs = [torch.zeros(n, device="cuda") for _ in range(4)]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        tps.ar_reduce(src_t, outs, dst_dtype="f32", wire_dtype="f16", stream=s)
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    for o in outs:
        assert_same(to_host(o, "f32"), exp, "f32", "graph replay")
    # replay again on new inputs written into the same buffers
    srcs2 = srcs_for(12, 4, n, "f32")
    for t, a in zip(src_t, srcs2):
        t.copy_(to_device(a, "f32"))
    g.replay()
    torch.cuda.synchronize()
    assert_same(to_host(outs[3], "f32"), expect(srcs2, "f32", "f16"), "f32", "second replay")


def test_host_entry_point(ctx):
    """ar_reduce_host: pinned host partials in, host results out."""
    w = W.WORKLOADS["tp_small"]
    srcs = W.generate(w)
    ctx.ensure(w.R, w.nelem)
    exp = expect(srcs, w.dst, w.wire)
    h_srcs = [torch.from_numpy(s).pin_memory() for s in srcs]
    h_dsts = [torch.empty(w.nelem, dtype=torch.float32).pin_memory() for _ in range(w.n_dsts)]
    d_srcs = [torch.empty(w.nelem, device="cuda") for _ in range(w.R)]
    d_dsts = [torch.empty(w.nelem, device="cuda") for _ in range(w.n_dsts)]
    tps.ar_reduce_host(h_srcs, h_dsts, d_srcs, d_dsts, dst_dtype="f32", wire_dtype=w.wire)
    torch.cuda.synchronize()
    for h in h_dsts:
        assert_same(h.numpy(), exp, "f32", "host entry")


@pytest.mark.parametrize("dst", TYPES)
@pytest.mark.parametrize("R", [2, 5])
def test_sixteen_but_not_32_byte_aligned(ctx, dst, R):
    """Pointers 16-byte aligned but not 32-byte aligned take the 16-byte
    vectors of the bandwidth variant; same bits."""
    n = 100_003
    shift = 16 // (4 if dst == "f32" else 2)  # one 16-byte step, in elements
    srcs = srcs_for(R + 40, R, n, dst)
    exp = expect(srcs, dst, "f16")
    outs, backs = run(ctx, srcs, 2, dst, "f16", variant="bandwidth", src_offsets=[shift] + [0] * (R - 1),
                      dst_offsets=[0, shift], pad=64)
    for o in outs:
        assert_same(o, exp, dst, "16-byte aligned")
    check_guards(backs)


@pytest.mark.parametrize("per_sm", [1, 2, 3])
@pytest.mark.parametrize("dst,R", [("f32", 2), ("f32", 8), ("bf16", 4)])
def test_persistent_grid_option(ctx, per_sm, dst, R):
    """A persistent bandwidth grid (CTAs sweep the tensors in rounds) gives
    the same bits as the covering grid."""
    n = 1_000_003
    srcs = srcs_for(per_sm * 7 + R, R, n, dst)
    exp = expect(srcs, dst, "bf16")
    ctx.ensure(R, n)
    tps.ar_set_option("bw_blocks_per_sm", per_sm)
    try:
        outs, _ = run(ctx, srcs, 2, dst, "bf16", variant="bandwidth")
    finally:
        tps.ar_set_option("bw_blocks_per_sm", 0)
    for o in outs:
        assert_same(o, exp, dst, f"persistent per_sm={per_sm}")


@pytest.mark.parametrize("chunk_bytes", [4096, 65536, 1 << 22])
@pytest.mark.parametrize("dst,wire,n", [("f32", "bf16", 1_000_003), ("bf16", "bf16", 777_777), ("f32", "f16", 4099)])
def test_host_entry_chunked_pipeline(ctx, chunk_bytes, dst, wire, n):
    """ar_reduce_host in chunks over its own streams: same bits as the
    oracle for every chunk size (small chunks hit the 64-chunk cap), on a
    non-default caller stream, twice in a row on the same staging buffers."""
    R, n_dsts = 3, 2
    ctx.ensure(R, n)
    tps.ar_set_option("host_chunk_bytes", chunk_bytes)
    try:
        stream = torch.cuda.Stream()
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dst]
        d_srcs = [torch.empty(n, dtype=tdt, device="cuda") for _ in range(R)]
        d_dsts = [torch.empty(n, dtype=tdt, device="cuda") for _ in range(n_dsts)]
        for call in range(2):
            srcs = srcs_for(chunk_bytes + call, R, n, dst)
            exp = expect(srcs, dst, wire)
            h_srcs = [torch.from_numpy(s.view(np.int16) if s.dtype == np.uint16 else s).pin_memory() for s in srcs]
            h_dsts = [torch.empty(n, dtype=h_srcs[0].dtype).pin_memory() for _ in range(n_dsts)]
            tps.ar_reduce_host(h_srcs, h_dsts, d_srcs, d_dsts, nelem=n, dst_dtype=dst, wire_dtype=wire, stream=stream)
            stream.synchronize()
            for h in h_dsts:
                assert_same(h.numpy().view(np.uint32 if dst == "f32" else np.uint16), exp, dst,
                            f"host pipeline chunk={chunk_bytes} call={call}")
    finally:
        tps.ar_set_option("host_chunk_bytes", 4 << 20)


def test_host_entry_in_place(ctx):
    """Device staging destination equal to a device staging source."""
    R, n = 2, 300_001
    ctx.ensure(R, n)
    srcs = srcs_for(99, R, n, "f32")
    exp = expect(srcs, "f32", "bf16")
    h_srcs = [torch.from_numpy(s).pin_memory() for s in srcs]
    h_dst = torch.empty(n, dtype=torch.float32).pin_memory()
    d_srcs = [torch.empty(n, device="cuda") for _ in range(R)]
    tps.ar_set_option("host_chunk_bytes", 65536)
    try:
        tps.ar_reduce_host(h_srcs, [h_dst], d_srcs, [d_srcs[1]], nelem=n, dst_dtype="f32", wire_dtype="bf16")
        torch.cuda.synchronize()
    finally:
        tps.ar_set_option("host_chunk_bytes", 4 << 20)
    assert_same(h_dst.numpy(), exp, "f32", "host in place")
    assert_same(to_host(d_srcs[1], "f32"), exp, "f32", "device destination")


def test_host_entry_refuses_partly_overlapping_host_buffers(ctx):
    """Staged ar_reduce_host: a host destination that partly overlaps a host
    source (its copy back of one chunk would overwrite source bytes a later
    chunk still has to copy in), or another host destination, is refused
    before anything is enqueued; exactly a source (in place) is allowed."""
    R, n = 2, 300_001
    ctx.ensure(R, n)
    tps.ar_set_option("host_chunk_bytes", 65536)
    try:
        back = torch.from_numpy(srcs_for(77, 1, 3 * n, "f32")[0]).pin_memory()
        before = back.clone()
        h_srcs = [back[:n], back[2 * n:]]
        d_srcs = [torch.full((n,), 7.0, device="cuda") for _ in range(R)]
        d_dst, d_dst2 = torch.full((n,), 7.0, device="cuda"), torch.full((n,), 7.0, device="cuda")
        other = torch.zeros(2 * n).pin_memory()
        for h_dsts in ([back[n // 2:n // 2 + n]], [back[1:n + 1]], [other[:n], other[n // 3:n // 3 + n]]):
            with pytest.raises(tps.ARError) as e:
                tps.ar_reduce_host(h_srcs, h_dsts, d_srcs, [d_dst, d_dst2][:len(h_dsts)], nelem=n,
                                   dst_dtype="f32", wire_dtype="bf16")
            assert e.value.status == 5
        torch.cuda.synchronize()
        assert torch.equal(back.view(torch.int32), before.view(torch.int32)) and not other.any()  # NaNs inside
        assert all((d == 7.0).all() for d in d_srcs + [d_dst, d_dst2])
        exp = expect([h.numpy().copy() for h in h_srcs], "f32", "bf16")
        tps.ar_reduce_host(h_srcs, [h_srcs[1]], d_srcs, [d_dst], nelem=n, dst_dtype="f32", wire_dtype="bf16")
        torch.cuda.synchronize()
    finally:
        tps.ar_set_option("host_chunk_bytes", 4 << 20)
    assert_same(h_srcs[1].numpy(), exp, "f32", "staged host in place")


@pytest.mark.parametrize("dst,wire,R,n", [("f32", "bf16", 2, 1_000_003), ("bf16", "bf16", 4, 333_333),
                                          ("f32", "f16", 8, 4099)])
def test_host_entry_direct(ctx, dst, wire, R, n):
    """ar_reduce_host without staging buffers: the kernel reads the pinned
    host partials and writes the pinned host results itself."""
    ctx.ensure(R, n)
    srcs = srcs_for(R * 13 + n, R, n, dst)
    exp = expect(srcs, dst, wire)
    h_srcs = [torch.from_numpy(s.view(np.int16) if s.dtype == np.uint16 else s).pin_memory() for s in srcs]
    h_dsts = [torch.empty(n, dtype=h_srcs[0].dtype).pin_memory() for _ in range(2)]
    stream = torch.cuda.Stream()
    tps.ar_reduce_host(h_srcs, h_dsts, nelem=n, dst_dtype=dst, wire_dtype=wire, stream=stream)
    stream.synchronize()
    for h in h_dsts:
        assert_same(h.numpy().view(np.uint32 if dst == "f32" else np.uint16), exp, dst, "direct host")


@pytest.mark.parametrize("n", [4099, 3_000_017])  # the latency and the bandwidth launch
def test_device_entry_point_on_pinned_host_memory(ctx, n):
    """ar_reduce given pinned host buffers as its device pointers (the GPU
    reaches them over the CPU-GPU link): two calls back to back on a created
    stream, so the second launches as a programmatic dependent and its first
    wave prefetches before it waits; both give the oracle's bits."""
    R = 3
    ctx.ensure(R, n)
    srcs = srcs_for(n + 5, R, n, "f32")
    exp = expect(srcs, "f32", "bf16")
    h_srcs = [torch.from_numpy(s).pin_memory() for s in srcs]
    h_dsts = [torch.full((n,), float("nan")).pin_memory() for _ in range(2)]
    stream = torch.cuda.Stream()
    for k in range(2):
        tps.ar_reduce_variant([h.data_ptr() for h in h_srcs], [h_dsts[k].data_ptr()], "auto", nelem=n,
                              dst_dtype="f32", wire_dtype="bf16", stream=stream)
    stream.synchronize()
    for h in h_dsts:
        assert_same(h.numpy(), exp, "f32", f"pinned host buffers n={n}")


@pytest.mark.parametrize("offsets,want", [((1, 1, 1), "bandwidth"), ((1, 2, 3), "scalar")])
def test_host_entry_direct_unaligned_and_in_place(ctx, offsets, want):
    """Pinned buffers off 16-byte alignment: one shared offset keeps the
    vector kernel, different offsets take the element-wise one."""
    R, n = 3, 50_001
    ctx.ensure(R, n)
    srcs = srcs_for(5150, R, n, "f32")
    exp = expect(srcs, "f32", "f16")
    backs = [torch.empty(n + 4, dtype=torch.float32).pin_memory() for _ in range(R)]
    assert all(b.data_ptr() % 16 == 0 for b in backs)
    h_srcs = [b[o:o + n] for b, o in zip(backs, offsets)]  # 4 * o bytes off 16-byte alignment
    for h, s in zip(h_srcs, srcs):
        h.copy_(torch.from_numpy(s))
    tps.ar_reduce_host(h_srcs, [h_srcs[2]], nelem=n, dst_dtype="f32", wire_dtype="f16")
    torch.cuda.synchronize()
    assert tps.ar_query("last_variant") == tps.ar.VARIANTS[want]
    assert_same(h_srcs[2].numpy(), exp, "f32", "direct, unaligned, in place")


def test_host_entry_direct_rejects_pageable_memory(ctx):
    ctx.ensure(2, 1024)
    a = np.ones(1024, dtype=np.float32)
    b = np.ones(1024, dtype=np.float32)
    out = np.full(1024, 7.0, dtype=np.float32)
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce_host([a, b], [out], nelem=1024, dst_dtype="f32", wire_dtype="bf16")
    assert e.value.status == 1
    assert (out == 7.0).all()


@pytest.mark.parametrize("wire", ["bf16", "f16"])
def test_kernel_casts_on_structured_patterns(ctx, wire):
    """R = 1 through the kernels is the wire round-trip: every sign,
    exponent and kept-fraction pattern crossed with the tie-deciding low bits
    (the inputs the CPU pins check the oracle on), through the bandwidth and
    latency paths, against the oracle."""
    from tests.test_oracle_casts import _structured_inputs
    x = _structured_inputs(wire)
    exp = oracle.reduce([x], 1, "f32", wire)[0]
    for v in ("bandwidth", "latency"):
        outs, _ = run(ctx, [x], 1, "f32", wire, variant=v)
        assert_same(outs[0], exp, "f32", f"casts {wire} via {v}")


def test_concurrent_calls_from_two_threads(ctx):
    """Two host threads enqueue reductions on their own streams at once; the
    context is shared and every result is right."""
    import threading
    R, n = 3, 200_003
    ctx.ensure(R, n)
    cases = []
    for k in range(2):
        srcs = srcs_for(300 + k, R, n, "f32")
        cases.append((srcs, expect(srcs, "f32", "f16"), [to_device(s, "f32") for s in srcs],
                      torch.empty(n, device="cuda"), torch.cuda.Stream()))
    errors = []

    def worker(k):
        try:
            _, _, s_t, out, stream = cases[k]
            for _ in range(50):
                tps.ar_reduce(s_t, [out], dst_dtype="f32", wire_dtype="f16", stream=stream)
            stream.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for srcs, exp, _, out, _ in cases:
        assert_same(to_host(out, "f32"), exp, "f32", "concurrent")


def test_host_calls_with_pageable_memory_beside_device_calls(ctx):
    """Three threads at once: two run staged ar_reduce_host calls on pageable
    (numpy) buffers, whose copies block the calling thread, each on its own
    stream and staging buffers; the third runs ar_reduce on device buffers.
    The staged calls take turns on the pipeline, nothing deadlocks, and every
    result is right."""
    import threading
    R, n = 3, 300_007
    ctx.ensure(R, n)
    errors, host_cases = [], []
    for k in range(2):
        srcs = srcs_for(700 + k, R, n, "f32")
        host_cases.append((srcs, expect(srcs, "f32", "bf16"), [np.full(n, np.nan, np.float32) for _ in range(2)],
                           [torch.empty(n, device="cuda") for _ in range(R)],
                           [torch.empty(n, device="cuda") for _ in range(2)], torch.cuda.Stream()))
    dsrcs = srcs_for(709, R, n, "f32")
    dexp = expect(dsrcs, "f32", "bf16")
    d_t = [to_device(a, "f32") for a in dsrcs]
    d_out = torch.empty(n, device="cuda")
    d_stream = torch.cuda.Stream()

    def host_worker(k):
        try:
            srcs, _, outs, ds, dd, stream = host_cases[k]
            for _ in range(10):
                tps.ar_reduce_host(srcs, outs, ds, dd, nelem=n, dst_dtype="f32", wire_dtype="bf16", stream=stream)
            stream.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    def device_worker():
        try:
            for _ in range(200):
                tps.ar_reduce(d_t, [d_out], dst_dtype="f32", wire_dtype="bf16", stream=d_stream)
            d_stream.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=host_worker, args=(k,)) for k in range(2)]
    threads.append(threading.Thread(target=device_worker))
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors
    for _, exp, outs, _, _, _ in host_cases:
        for o in outs:
            assert_same(o, exp, "f32", "staged, pageable, from a thread")
    assert_same(to_host(d_out, "f32"), dexp, "f32", "device calls beside host calls")


@pytest.mark.parametrize("wire", ["bf16", "f16"])
def test_kernel_casts_exhaustive(ctx, wire):
    """Every float32 bit pattern through the kernel with R = 1 (the wire
    round-trip, where the kernel's packed round-to-nearest-even converts
    decide every bit) against the oracle, in chunks of 2^26; the oracle runs
    in parallel threads on the host."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    chunk = 1 << 26
    ctx.ensure(1, chunk)
    d_in = torch.empty(chunk, dtype=torch.float32, device="cuda")
    d_out = torch.empty_like(d_in)
    h_out = torch.empty(chunk, dtype=torch.float32).pin_memory()
    nthreads = os.cpu_count() or 8
    part = chunk // nthreads
    with ThreadPoolExecutor(nthreads) as pool:
        for start in range(0, 1 << 32, chunk):
            x = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
            d_in.copy_(torch.from_numpy(x))
            tps.ar_reduce([d_in], [d_out], dst_dtype="f32", wire_dtype=wire)
            h_out.copy_(d_out)
            exp = np.empty(chunk, dtype=np.float32)
            list(pool.map(lambda k: oracle.reduce([x], 1, "f32", wire, begin=k * part,
                                                  end=chunk if k == nthreads - 1 else (k + 1) * part,
                                                  out=[exp]), range(nthreads)))
            assert_same(h_out.numpy(), exp, "f32", f"{wire} chunk {start:#x}")


@pytest.mark.parametrize("variant", ["auto", "bandwidth", "latency", "scalar", "tma"])
def test_sixteen_ranks_sixteen_destinations(ctx, variant):
    """The largest call the ABI allows: R = 16 and n_dsts = 16."""
    n = 65_539
    srcs = srcs_for(16161, 16, n, "bf16")
    exp = expect(srcs, "bf16", "f16")
    outs, backs = run(ctx, srcs, 16, "bf16", "f16", variant=variant, pad=32)
    for d, o in enumerate(outs):
        assert_same(o, exp, "bf16", f"R=16 n_dsts=16 {variant} dst={d}")
    check_guards(backs)


def test_more_than_2_31_elements(ctx):
    """64-bit indexing: 2^31 + 7 bf16 elements per buffer (4 GiB each), two
    sources and one destination; every element is compared with the oracle
    (run on every host core)."""
    n = (1 << 31) + 7
    ctx.ensure(2, n)
    # cheap deterministic finite bf16 patterns: exponent fields 100..140, any sign and fraction
    base = np.arange(n, dtype=np.uint32)
    a = ((base * np.uint32(2654435761)) >> np.uint32(16)).astype(np.uint16)
    b = ((base * np.uint32(40503)) >> np.uint32(8)).astype(np.uint16)
    del base
    for x in (a, b):
        e = (np.uint16(100) + (x >> np.uint16(7)) % np.uint16(41)).astype(np.uint16)
        x[:] = (x & np.uint16(0x807F)) | (e << np.uint16(7))
    d_a, d_b = to_device(a, "bf16"), to_device(b, "bf16")
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    tps.ar_reduce([d_a, d_b], [out], nelem=n, dst_dtype="bf16", wire_dtype="f16")
    torch.cuda.synchronize()
    del d_a, d_b
    got = to_host(out, "bf16")
    del out
    assert_same(got, whole.reduce([a, b], "bf16", "f16"), "bf16", "2^31 + 7 elements")


@pytest.mark.parametrize("grid", [1, 3, 152])
def test_tma_grids_and_status(ctx, grid):
    """The bulk-copy variant on 1, 3 and 152 CTAs (many tiles per CTA, all
    three stages cycling) gives the oracle's bits, and none of its bounded
    waits ran out."""
    tps.ar_init(3, 1 << 20)
    ctx.R = None
    tps.ar_set_option("device_status", 0)
    n = 3_000_017
    srcs = srcs_for(grid + 500, 3, n, "f32")
    outs, backs = run(ctx, srcs, 2, "f32", "bf16", variant="tma", grid=grid, pad=64)
    exp = expect(srcs, "f32", "bf16")
    for o in outs:
        assert_same(o, exp, "f32", f"tma grid={grid}")
    check_guards(backs)
    assert tps.ar_query("device_status") == 0


@pytest.mark.parametrize("stages,tile,ctas", [(2, 1024, 1), (8, 1024, 4), (4, 32768, 1)])
def test_tma_knobs(ctx, monkeypatch, stages, tile, ctas):
    """The bulk-copy variant at the edges of its settings (read at ar_init)."""
    monkeypatch.setenv("AR_TMA_STAGES", str(stages))
    monkeypatch.setenv("AR_TMA_TILE", str(tile))
    monkeypatch.setenv("AR_TMA_CTAS_PER_SM", str(ctas))
    n, R = 1_234_567, 4
    tps.ar_init(R, n)
    ctx.R = None
    try:
        tps.ar_set_option("device_status", 0)
        srcs = srcs_for(stages * 100 + ctas, R, n, "bf16")
        src_t = [to_device(s, "bf16") for s in srcs]
        dst_t = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        tps.ar_reduce_variant(src_t, dst_t, "tma", nelem=n, dst_dtype="bf16", wire_dtype="f32")
        torch.cuda.synchronize()
        exp = expect(srcs, "bf16", "f32")
        for d in dst_t:
            assert_same(to_host(d, "bf16"), exp, "bf16", f"tma stages={stages} tile={tile} ctas={ctas}")
        assert tps.ar_query("device_status") == 0
    finally:
        monkeypatch.undo()
        tps.ar_init(R, n)


def test_tma_bounded_wait_runs_out_reports_and_context_survives(ctx):
    """Failure detection without a GPU fault: the test hook keeps one tile's
    data from ever arriving, the waiting CTA gives up after its bound,
    the host reads the error from the status word, and the same context
    then reduces correctly again."""
    R, n = 2, 1_000_003
    tps.ar_init(R, n)
    ctx.R = None
    srcs = srcs_for(777, R, n, "f32")
    src_t = [to_device(s, "f32") for s in srcs]
    out = torch.empty(n, device="cuda")
    tps.ar_set_option("device_status", 0)
    tps.ar_set_option("tma_drop_tile", 3)
    try:
        tps.ar_reduce_variant(src_t, [out], "tma", dst_dtype="f32", wire_dtype="bf16")
        torch.cuda.synchronize()  # ends: the wait is bounded
        assert tps.ar_query("device_status") & 1
    finally:
        tps.ar_set_option("tma_drop_tile", -1)
    tps.ar_set_option("device_status", 0)
    tps.ar_reduce_variant(src_t, [out], "tma", dst_dtype="f32", wire_dtype="bf16")
    torch.cuda.synchronize()
    assert tps.ar_query("device_status") == 0
    assert_same(to_host(out, "f32"), expect(srcs, "f32", "bf16"), "f32", "after a timed-out launch")


def test_dependent_launch_still_honours_event_waits(ctx):
    """The vector kernels launch as programmatic dependents of the kernel
    before them on the stream.  A cross-stream event wait between the two
    must still hold: the second reduction reads partials that another
    stream writes only after a delay."""
    n = 1 << 20
    ctx.ensure(2, n)
    side, main = torch.cuda.Stream(), torch.cuda.Stream()
    a = torch.zeros(n, device="cuda")
    b = torch.zeros(n, device="cuda")
    warm = torch.ones(n, device="cuda")
    out1 = torch.empty(n, device="cuda")
    out2 = torch.empty(n, device="cuda")
    torch.cuda.synchronize()
    ready = torch.cuda.Event()
    with torch.cuda.stream(side):
        torch.cuda._sleep(20_000_000)  # a bounded delay (about 10 ms) before the partials are written
        a.fill_(1.5)
        b.fill_(2.25)
        ready.record(side)
    tps.ar_reduce([warm, warm], [out1], wire_dtype="f32", stream=main)  # the kernel before, on `main`
    main.wait_event(ready)
    tps.ar_reduce([a, b], [out2], wire_dtype="f32", stream=main)
    torch.cuda.synchronize()
    assert tps.ar_query("last_variant") == tps.ar.VARIANTS["latency"]
    assert (out1 == 2.0).all()
    assert (out2 == 3.75).all()


def test_dependent_launch_after_a_copy_on_the_same_stream(ctx):
    """Kernel, then a host-to-device copy, then a reduction of the copied
    partials, all on one stream: the reduction sees the copy."""
    n = 1 << 22
    ctx.ensure(2, n)
    main = torch.cuda.Stream()
    warm = torch.ones(n, device="cuda")
    a = torch.zeros(n, device="cuda")
    host = torch.full((n,), 4.0).pin_memory()
    out1 = torch.empty(n, device="cuda")
    out2 = torch.empty(n, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(main):
        tps.ar_reduce([warm, warm], [out1], wire_dtype="f32", stream=main)
        a.copy_(host, non_blocking=True)
        tps.ar_reduce([a, warm], [out2], wire_dtype="f32", stream=main)
    torch.cuda.synchronize()
    assert (out1 == 2.0).all()
    assert (out2 == 5.0).all()


@pytest.mark.parametrize("pdl", ["0", "1"])
def test_plain_and_dependent_launches_give_the_same_bits(ctx, pdl, monkeypatch):
    """AR_PDL=0 launches every kernel plainly; the bits do not change."""
    monkeypatch.setenv("AR_PDL", pdl)
    tps.ar_init(3, 1 << 20)
    ctx.R = None  # the next test re-initialises with its own limits (and without the variable)
    n = 300_007
    srcs = srcs_for(4242, 3, n, "f32")
    exp = expect(srcs, "f32", "bf16")
    stream = torch.cuda.Stream()  # a created stream: the default streams always launch plainly
    for v in VARIANTS:
        d_srcs = [to_device(s, "f32") for s in srcs]
        d_dsts = [torch.empty(n, device="cuda") for _ in range(2)]
        torch.cuda.synchronize()
        tps.ar_reduce_variant(d_srcs, d_dsts, v, dst_dtype="f32", wire_dtype="bf16", stream=stream)
        tps.ar_reduce_variant(d_srcs, d_dsts, v, dst_dtype="f32", wire_dtype="bf16", stream=stream)
        torch.cuda.synchronize()
        for d in d_dsts:
            assert_same(to_host(d, "f32"), exp, "f32", f"AR_PDL={pdl} variant={v}")


@pytest.mark.parametrize("prefetch", ["0", "1"])
@pytest.mark.parametrize("n", [100_003, 3_000_017])  # the latency and the bandwidth launch
def test_chained_reductions_see_the_previous_results(ctx, prefetch, n, monkeypatch):
    """Each reduction sums the previous one's output with a new partial; the
    six launches run back to back on one created stream inside a CUDA graph,
    each a programmatic dependent of the one before, which (AR_L2_PREFETCH=1,
    the default) asks L2 for its sources before it waits for that kernel.
    Every step must read the previous step's final bits: the chain equals the
    oracle's chain, with the prefetch on and off."""
    monkeypatch.setenv("AR_L2_PREFETCH", prefetch)
    tps.ar_init(2, n)
    ctx.R = None  # the next test re-initialises with its own limits (and without the variable)
    steps = 6
    parts = srcs_for(n + int(prefetch), steps + 1, n, "f32")
    exp, prev = [], parts[0]
    for k in range(1, steps + 1):
        prev = expect([prev, parts[k]], "f32", "bf16")
        exp.append(prev)
    d_parts = [to_device(a, "f32") for a in parts]
    outs = [torch.empty(n, device="cuda") for _ in range(steps)]
    stream = torch.cuda.Stream()

    def chain(s):
        src = d_parts[0]
        for k in range(steps):
            tps.ar_reduce([src, d_parts[k + 1]], [outs[k]], dst_dtype="f32", wire_dtype="bf16", stream=s)
            src = outs[k]

    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        chain(stream)
    for o in outs:
        o.view(torch.int32).fill_(0x7FC00001)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for k in range(steps):
        assert_same(to_host(outs[k], "f32"), exp[k], "f32", f"step {k + 1} AR_L2_PREFETCH={prefetch}")


@pytest.mark.parametrize("prefetch", ["0", "1"])
def test_prefetch_on_and_off_give_the_same_bits_for_every_variant(ctx, prefetch, monkeypatch):
    """AR_L2_PREFETCH=0 turns the first wave's L2 prefetch off; every variant
    gives the oracle's bits either way, two launches back to back on a
    created stream (the second a programmatic dependent of the first)."""
    monkeypatch.setenv("AR_L2_PREFETCH", prefetch)
    tps.ar_init(3, 1 << 20)
    ctx.R = None  # the next test re-initialises with its own limits (and without the variable)
    n = 300_007
    srcs = srcs_for(4343, 3, n, "bf16")
    exp = expect(srcs, "bf16", "f16")
    stream = torch.cuda.Stream()
    for v in VARIANTS:
        d_srcs = [to_device(s, "bf16") for s in srcs]
        d_dsts = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        torch.cuda.synchronize()
        for _ in range(2):
            tps.ar_reduce_variant(d_srcs, d_dsts, v, dst_dtype="bf16", wire_dtype="f16", stream=stream)
        torch.cuda.synchronize()
        for d in d_dsts:
            assert_same(to_host(d, "bf16"), exp, "bf16", f"AR_L2_PREFETCH={prefetch} variant={v}")


@pytest.mark.parametrize("variant", ["auto", "latency", "bandwidth", "scalar"])
def test_prepared_call_gives_the_same_bits(ctx, variant):
    n = 50_003
    ctx.ensure(3, n)
    srcs = srcs_for(909, 3, n, "bf16")
    exp = expect(srcs, "bf16", "f16")
    d_srcs = [to_device(s, "bf16") for s in srcs]
    d_dsts = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    call = tps.PreparedReduce(d_srcs, d_dsts, wire_dtype="f16", variant=variant)
    for _ in range(3):  # repeatable
        for d in d_dsts:
            d.fill_(7)
        call()
        torch.cuda.synchronize()
        for d in d_dsts:
            assert_same(to_host(d, "bf16"), exp, "bf16", f"prepared {variant}")
