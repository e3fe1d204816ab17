"""GPU parity of the extended layouts (ar_reduce_ex: row strides, inactive
ranks, residual and row-broadcast bias) and of the wire pack, against the
oracle, bit for bit (any NaN matches any NaN)."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import tensor_partial_sum_gb300 as tps
from tests.gpu_util import TORCH_DTYPE, to_device, to_host
from tests.libcasts import assert_same, lib_round
from tests.test_oracle_fold import edgy_f32

pytestmark = pytest.mark.gpu

TYPES = ["f32", "f16", "bf16"]
PAIRS = list(itertools.product(TYPES, TYPES))
ES = {"f32": 4, "f16": 2, "bf16": 2}


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_partial_sum_gb300 import build
    build.build()
    yield
    tps.ar_free()


def srcs_for(seed, R, n, dst):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [lib_round(dst, edgy_f32(rng, n)) for _ in range(R)]


def strided_device(flat_rows, ne0, ne1, stride_elems, dst, lead=0, fill=0x5A):
    """Device buffer holding ne1 rows at stride_elems (elements), starting
    `lead` elements into a poisoned allocation; returns (view start tensor,
    backing bytes)."""
    es = ES[dst]
    total = lead + (ne1 - 1) * stride_elems + ne0 if ne1 else lead + 1
    back = torch.full((total * es + 64,), fill, dtype=torch.uint8, device="cuda")
    t = back[:total * es].view(TORCH_DTYPE[dst])
    if flat_rows is not None:
        dev = to_device(flat_rows, dst)
        for j in range(ne1):
            t[lead + j * stride_elems: lead + j * stride_elems + ne0].copy_(dev[j * ne0:(j + 1) * ne0])
    return t[lead:], back


def rows_of(t, ne0, ne1, stride_elems, dst):
    h = to_host(t, dst)
    return np.concatenate([h[j * stride_elems: j * stride_elems + ne0] for j in range(ne1)]) if ne1 else h[:0]


def run_ex(R, ne0, ne1, dst, wire, seed, src_pad=None, dst_pad=(0,), lead=0, inactive=(), residual=None,
           bias=False, n_dsts=1, res_pad=None):
    """Run ar_reduce_ex and the oracle on the same strided inputs."""
    es = ES[dst]
    src_pad = src_pad or [0] * R
    srcs = srcs_for(seed, R, ne0 * ne1, dst)
    tps.ar_init(R, max(1, ne0 * ne1))
    s_t = []
    for r in range(R):
        if r in inactive:
            s_t.append(None)
            continue
        t, _ = strided_device(srcs[r], ne0, ne1, ne0 + src_pad[r], dst, lead=lead)
        s_t.append(t)
    d_t, d_backs = [], []
    pads = list(dst_pad) + [0] * (n_dsts - len(dst_pad))
    for d in range(n_dsts):
        t, back = strided_device(None, ne0, ne1, ne0 + pads[d], dst, lead=lead)
        d_t.append(t)
        d_backs.append(back)
    res_t = res_np = None
    res_stride = None
    if residual:
        res_np = srcs_for(seed + 1, 1, ne0 if bias else ne0 * ne1, dst)[0]
        V = 16 // es
        rpad = res_pad if res_pad is not None else (V if ne0 % V == 0 else 3)  # aligned rows stay aligned
        res_t, _ = strided_device(res_np, ne0, 1 if bias else ne1, ne0 + (0 if bias else rpad), dst, lead=lead)
        res_stride = 0 if bias else (ne0 + rpad) * es
    layout = tps.make_layout(ne0, ne1, src_row_bytes=[(ne0 + p) * es for p in src_pad],
                             dst_row_bytes=[(ne0 + p) * es for p in pads], residual=res_t,
                             residual_row_bytes=res_stride, inactive=inactive)
    tps.ar_reduce_ex(s_t, d_t, layout, dst, wire)
    torch.cuda.synchronize()
    holes = [None if r in inactive else s for r, s in enumerate(srcs)]
    exp = oracle.reduce_2d(holes, 1, dst, wire, ne0, ne1, inactive=inactive, residual=res_np,
                           residual_stride=0 if bias else None)[0]
    for d, t in enumerate(d_t):
        assert_same(rows_of(t, ne0, ne1, ne0 + pads[d], dst), exp, dst,
                    f"ex R={R} {ne0}x{ne1} inactive={inactive} residual={residual} bias={bias} d={d}")
    return d_backs


@pytest.mark.parametrize("dst,wire", PAIRS)
@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_packed_2d_all_pairs(dst, wire, R):
    run_ex(R, 4096 + 5, 7, dst, wire, seed=R * 3 + len(dst + wire), n_dsts=2)


@pytest.mark.parametrize("dst,wire", [("f32", "bf16"), ("bf16", "bf16"), ("f16", "f32")])
@pytest.mark.parametrize("ne0,ne1", [(1, 1), (3, 5), (7, 3), (8, 2), (64, 300), (1000, 3), (4097, 2),
                                     (100_000, 1)])
def test_shapes(dst, wire, ne0, ne1):
    run_ex(3, ne0, ne1, dst, wire, seed=ne0 + ne1, n_dsts=2)


@pytest.mark.parametrize("dst", TYPES)
@pytest.mark.parametrize("kind", ["aligned", "odd_strides", "odd_start"])
def test_row_strides(dst, kind):
    """Padded rows (ne0 = 777 leaves a ragged tail in every row): strides
    that are multiples of 16 bytes take the vector path with a per-row tail
    (after a per-row head when every buffer starts one element in), strides
    that differ modulo 16 bytes the element-wise path; the padding between
    rows is never written."""
    ne0, ne1, es = 777, 9, ES[dst]
    V = 16 // es
    base = (V - ne0 % V) % V
    if kind == "odd_strides":
        pads, lead = [1, 2, 3], 0
    else:
        pads, lead = [base + k * V for k in (1, 2, 3)], (1 if kind == "odd_start" else 0)
    backs = run_ex(3, ne0, ne1, dst, "bf16", seed=11, src_pad=pads, dst_pad=(pads[0], base), lead=lead, n_dsts=2)
    b = backs[0].cpu().numpy()
    stride = (ne0 + pads[0]) * es
    for j in range(ne1 - 1):
        gap = b[lead * es + j * stride + ne0 * es: lead * es + (j + 1) * stride]
        assert (gap == 0x5A).all(), "padding written"


@pytest.mark.parametrize("wire", TYPES)
@pytest.mark.parametrize("R", [2, 3])
def test_f32_32_byte_rows(wire, R):
    """f32 rows whose starts and strides are all multiples of 32 bytes take
    the 32-byte vector path (ne0 = 777 leaves a 1-element tail per row)."""
    ne0 = 777
    base = (8 - ne0 % 8) % 8
    run_ex(R, ne0, 11, "f32", wire, seed=91 + R, src_pad=[base + 8 * r for r in range(R)],
           dst_pad=(base, base + 8), inactive=(1,) if R == 3 else (), residual=True, n_dsts=2, res_pad=base + 16)


@pytest.mark.parametrize("dst,wire", PAIRS)
@pytest.mark.parametrize("inactive", [(0,), (1,), (0, 2), (0, 1, 2)])
def test_inactive_ranks(dst, wire, inactive):
    run_ex(3, 5000, 3, dst, wire, seed=21, inactive=inactive)


@pytest.mark.parametrize("dst,wire", PAIRS)
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("ne0", [4096, 4099])
def test_residual_and_bias(dst, wire, bias, ne0):
    """ne0 = 4096 keeps every row 16-byte aligned (vector path, residual row
    padded to a 16-byte stride); 4099 runs element by element."""
    run_ex(2, ne0, 6, dst, wire, seed=31, residual=True, bias=bias, n_dsts=2)


@pytest.mark.parametrize("R", [2, 5])
def test_residual_bias_inactive_strided_together(R):
    run_ex(R, 1031, 17, "f32", "f16", seed=41, src_pad=[4 * (r + 1) for r in range(R)], dst_pad=(12,),
           inactive=(1,), residual=True, bias=True)


def test_residual_in_place():
    """x = x + allreduce(partials): the destination is the residual."""
    R, ne0, ne1 = 2, 8192, 16
    srcs = srcs_for(51, R + 1, ne0 * ne1, "f32")
    tps.ar_init(R, ne0 * ne1)
    s_t = [to_device(s, "f32") for s in srcs[:R]]
    x = to_device(srcs[R], "f32")
    tps.ar_reduce_ex(s_t, [x], tps.make_layout(ne0, ne1, residual=x), "f32", "bf16")
    torch.cuda.synchronize()
    exp = oracle.reduce_2d(srcs[:R], 1, "f32", "bf16", ne0, ne1, residual=srcs[R])[0]
    assert_same(to_host(x, "f32"), exp, "f32", "residual in place")


def test_ex_packed_equals_ar_reduce():
    """Without strides, residual or inactive ranks, ar_reduce_ex gives the
    bits ar_reduce gives."""
    R, n = 4, 1 << 20
    srcs = srcs_for(61, R, n, "bf16")
    tps.ar_init(R, n)
    s_t = [to_device(s, "bf16") for s in srcs]
    a = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    tps.ar_reduce(s_t, [a], dst_dtype="bf16", wire_dtype="f16")
    tps.ar_reduce_ex(s_t, [b], tps.make_layout(1024, 1024), "bf16", "f16")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_ex_errors_write_nothing():
    tps.ar_init(2, 1 << 16)
    a = torch.randn(4096, device="cuda")
    out = torch.full((4096,), 7.0, device="cuda")
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce_ex([a, a], [out], tps.make_layout(64, 64, src_row_bytes=[100, 256]), "f32", "bf16")
    assert e.value.status == 1
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce_ex([a, None], [out], tps.make_layout(64, 64), "f32", "bf16")  # NULL active rank
    assert e.value.status == 1
    with pytest.raises(tps.ARError) as e:
        tps.ar_reduce_ex([a, a], [a[8:]], tps.make_layout(64, 63), "f32", "bf16")
    assert e.value.status == 5
    torch.cuda.synchronize()
    assert (out == 7.0).all()


@pytest.mark.parametrize("dst,wire", PAIRS)
@pytest.mark.parametrize("n", [1, 7, 8, 9, 4099, 1_000_003])
def test_wire_pack(dst, wire, n):
    (x,) = srcs_for(n + 71, 1, n, dst)
    tps.ar_init(1, max(n, 1))
    src = to_device(x, dst)
    out = torch.empty(n, dtype=TORCH_DTYPE[wire], device="cuda")
    tps.ar_wire_pack(src, out, dst_dtype=dst, wire_dtype=wire)
    torch.cuda.synchronize()
    assert_same(to_host(out, wire), oracle.wire_pack(x, dst, wire), wire, f"pack {dst}->{wire} n={n}")


@pytest.mark.parametrize("dst,wire", [("f32", "bf16"), ("bf16", "f32"), ("f16", "bf16")])
def test_wire_pack_unaligned_and_in_place(dst, wire):
    n = 10_001
    (x,) = srcs_for(81, 1, n, dst)
    tps.ar_init(1, n)
    back = torch.zeros(n + 1, dtype=TORCH_DTYPE[dst], device="cuda")
    src = back[1:]
    src.copy_(to_device(x, dst))
    out_back = torch.zeros(n + 1, dtype=TORCH_DTYPE[wire], device="cuda")
    out = out_back[1:]
    tps.ar_wire_pack(src, out, dst_dtype=dst, wire_dtype=wire)
    torch.cuda.synchronize()
    exp = oracle.wire_pack(x, dst, wire)
    assert_same(to_host(out, wire), exp, wire, "pack unaligned")
    if ES[dst] == ES[wire]:
        tps.ar_wire_pack(src, src, dst_dtype=dst, wire_dtype=wire)
        torch.cuda.synchronize()
        assert_same(to_host(src.view(TORCH_DTYPE[wire]), wire), exp, wire, "pack in place")


@pytest.mark.parametrize("dst", TYPES)
@pytest.mark.parametrize("case", ["start", "odd_stride", "odd_stride_and_start", "residual", "bias",
                                  "inactive", "different_strides"])
def test_common_row_offset_takes_the_vector_path(dst, case):
    """Rows that all start at one offset from a vector boundary, or whose
    starts all move by the same odd stride, run the vector kernel with each
    row's head done element by element: same bits, padding intact.  Strides
    that differ modulo 16 bytes run element by element."""
    ne0, ne1, R, es = 1001, 13, 3, ES[dst]
    V = 16 // es
    lead, pads, res_pad, kw = 0, [V] * R, None, {}
    if case == "start":
        lead = V - 1
    elif case == "odd_stride":
        pads = [1] * R
    elif case == "odd_stride_and_start":
        pads, lead = [3] * R, 2
    elif case == "residual":
        pads, lead, res_pad, kw = [1] * R, 1, 1, dict(residual=True)
    elif case == "bias":  # a broadcast row needs strides that are multiples of 16 bytes
        pads, lead, kw = [(V - ne0 % V) % V] * R, 1, dict(residual=True, bias=True)
    elif case == "inactive":
        pads, lead, kw = [1] * R, 3, dict(inactive=(0,))
    else:
        pads = [1, 2, 3]
    backs = run_ex(R, ne0, ne1, dst, "bf16", seed=len(case) * 7 + es, src_pad=pads, dst_pad=(pads[0], pads[0]),
                   lead=lead, n_dsts=2, res_pad=res_pad, **kw)
    want = "scalar" if case == "different_strides" else "bandwidth"
    assert tps.ar_query("last_variant") == tps.ar.VARIANTS[want]
    for b in backs:
        b = b.cpu().numpy()
        stride = (ne0 + pads[0]) * es
        assert (b[:lead * es] == 0x5A).all(), "bytes before the first row written"
        for j in range(ne1 - 1):
            gap = b[lead * es + j * stride + ne0 * es: lead * es + (j + 1) * stride]
            assert (gap == 0x5A).all(), "padding written"
        assert (b[lead * es + (ne1 - 1) * stride + ne0 * es:] == 0x5A).all(), "bytes after the last row written"


@pytest.mark.parametrize("wire", TYPES)
def test_common_row_offset_f32_32_byte_path(wire):
    """f32 strides that agree modulo 32 bytes (here 1036 floats = 4144 bytes,
    16 modulo 32) with a start 3 floats off: the 32-byte kernel with a
    per-row head of 5 or 1 elements."""
    ne0 = 1030
    run_ex(2, ne0, 9, "f32", wire, seed=5, src_pad=[6, 6], dst_pad=(6,), lead=3, residual=True, res_pad=6)
    assert tps.ar_query("last_variant") == tps.ar.VARIANTS["bandwidth"]


@pytest.mark.parametrize("dst,wire", PAIRS)
@pytest.mark.parametrize("offs", [(1, 1), (3, 3), (1, 2), (2, 1), (5, 7), (0, 1)])
@pytest.mark.parametrize("n", [1, 6, 70_001])
def test_wire_pack_offsets(dst, wire, offs, n):
    """Source and wire buffers starting off a vector boundary: where skipping
    the same first elements aligns both, the vector kernel runs after an
    element-wise head, else the element-wise kernel; the bits are the same
    and nothing outside the wire buffer is written."""
    so, wo = offs
    (x,) = srcs_for(n + so * 10 + wo, 1, n, dst)
    tps.ar_init(1, n)
    back = torch.zeros(n + so, dtype=TORCH_DTYPE[dst], device="cuda")
    src = back[so:]
    src.copy_(to_device(x, dst))
    out_back = torch.full(((n + wo) * ES[wire] + 64,), 0x5A, dtype=torch.uint8, device="cuda")
    out = out_back[wo * ES[wire]:(n + wo) * ES[wire]].view(TORCH_DTYPE[wire])
    tps.ar_wire_pack(src, out, dst_dtype=dst, wire_dtype=wire)
    torch.cuda.synchronize()
    assert_same(to_host(out, wire), oracle.wire_pack(x, dst, wire), wire, f"pack offsets {offs}")
    b = out_back.cpu().numpy()
    assert (b[:wo * ES[wire]] == 0x5A).all() and (b[(n + wo) * ES[wire]:] == 0x5A).all()
    # the buffers' addresses decide the kernel: some head aligns both or none does
    a0, b0 = src.data_ptr(), out.data_ptr()
    fits = any((a0 + h * ES[dst]) % 16 == 0 and (b0 + h * ES[wire]) % max(16 // ES[dst] * ES[wire], 16) == 0
               for h in range(16 // ES[dst]))
    if fits:
        assert tps.ar_query("last_variant") == tps.ar.VARIANTS["bandwidth"]


def test_binding_refuses_rows_past_the_storage():
    """Rows of a strided view may use the storage past the view's own last
    element (padding), but not past the storage's end."""
    ne0, ne1, pad = 100, 4, 28
    tps.ar_init(2, ne0 * ne1)
    back = torch.zeros(ne1 * (ne0 + pad), device="cuda")
    rows = back.view(ne1, ne0 + pad)[:, :ne0]  # not contiguous; reaches the storage's end
    stride = [(ne0 + pad) * 4] * 2
    out = torch.zeros(ne0 * ne1, device="cuda")
    tps.ar_reduce_ex([rows, rows], [out], tps.make_layout(ne0, ne1, src_row_bytes=stride), "f32")
    torch.cuda.synchronize()
    tail = back[(ne0 + pad):]  # one row less of storage
    with pytest.raises(ValueError, match="source 0 reaches"):
        tps.ar_reduce_ex([tail, rows], [out], tps.make_layout(ne0, ne1, src_row_bytes=stride), "f32")
    with pytest.raises(ValueError, match="destination 0 reaches"):
        tps.ar_reduce_ex([rows, rows], [out[1:]], tps.make_layout(ne0, ne1), "f32")


@pytest.mark.parametrize("ne0,pad", [(8, 0), (13, 3)])
def test_more_rows_than_the_grid_holds(ne0, pad):
    """ne1 above 65 535 (the grid's y limit): CTAs stride over the rows; both
    the vector path (ne0 = 8, packed) and the element-wise one (ne0 = 13 with
    differing strides) cover every row."""
    run_ex(2, ne0, 70_001, "f32", "bf16", seed=ne0, src_pad=[pad, 2 * pad], dst_pad=(0,), residual=True,
           res_pad=0)


@pytest.mark.parametrize("prefetch", ["0", "1"])
def test_chained_in_place_updates_and_pack_see_the_previous_results(prefetch, monkeypatch):
    """x = x + reduce(partials_k) four times in place into the residual (the
    destination is the residual), then the wire pack of the result, all back
    to back on one created stream inside a CUDA graph: each launch is a
    programmatic dependent of the one before, whose output it reads, and
    (AR_L2_PREFETCH=1, the default) asks L2 for its operands before waiting
    for it.  Every step must read the previous step's final bits."""
    monkeypatch.setenv("AR_L2_PREFETCH", prefetch)
    ne0, ne1, R, steps = 4096, 1024, 2, 4
    n = ne0 * ne1
    tps.ar_init(R, n)
    x0 = srcs_for(7 + int(prefetch), 1, n, "f32")[0]
    parts = [srcs_for(100 * k + int(prefetch), R, n, "f32") for k in range(steps)]
    exp = x0
    for k in range(steps):
        exp = oracle.reduce_2d(parts[k], 1, "f32", "bf16", ne0, ne1, residual=exp)[0]
    exp_pack = oracle.wire_pack(exp, "f32", "bf16")
    x = to_device(x0, "f32")
    d_parts = [[to_device(a, "f32") for a in p] for p in parts]
    wire = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    lay = tps.make_layout(ne0, ne1, residual=x)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(steps):
            tps.ar_reduce_ex(d_parts[k], [x], lay, "f32", "bf16", stream=stream)
        tps.ar_wire_pack(x, wire, dst_dtype="f32", wire_dtype="bf16", stream=stream)
    x.copy_(to_device(x0, "f32"))
    wire.view(torch.int16).fill_(0x7FC1)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert_same(to_host(x, "f32"), exp, "f32", f"in-place chain AR_L2_PREFETCH={prefetch}")
    assert_same(to_host(wire, "bf16"), exp_pack, "bf16", f"pack after the chain AR_L2_PREFETCH={prefetch}")
