"""Pins for the oracle's 2-D reduction (row strides, inactive ranks,
residual / row-broadcast bias) and its wire pack (CPU only).

Each pin ties orc_reduce_2d to something it does not share code with: the
1-D oracle's separate loop, the pages' own semantics restated (inactive
shards are zeroed tensors, ggml-cuda allreduce.cu, ggml_cuda_ar_allreduce),
and library casts with numpy float32 adds."""
import itertools

import numpy as np
import pytest

import oracle
from tests.libcasts import assert_same, lib_round, lib_widen
from tests.test_oracle_fold import edgy_f32

TYPES = ["f32", "f16", "bf16"]
PAIRS = list(itertools.product(TYPES, TYPES))
ES = {"f32": 4, "f16": 2, "bf16": 2}


def srcs_for(seed, R, n, dst):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [lib_round(dst, edgy_f32(rng, n)) for _ in range(R)]


def lib_fold_f32(srcs, dst, wire):
    acc = None
    for s in srcs:
        w = lib_widen(wire, lib_round(wire, lib_widen(dst, s)))
        with np.errstate(over="ignore", invalid="ignore"):
            acc = w.copy() if acc is None else (acc + w).astype(np.float32)
    return acc


def embed(rows, ne0, stride_elems, seed):
    """Rows of ne0 elements placed at a row stride, padding filled with noise."""
    ne1 = rows.size // ne0
    rng = np.random.Generator(np.random.PCG64(seed))
    flat = rng.integers(0, 1 << 16, (ne1 - 1) * stride_elems + ne0).astype(rows.dtype)
    for j in range(ne1):
        flat[j * stride_elems: j * stride_elems + ne0] = rows[j * ne0:(j + 1) * ne0]
    return flat


def extract(flat, ne0, ne1, stride_elems):
    return np.concatenate([flat[j * stride_elems: j * stride_elems + ne0] for j in range(ne1)])


@pytest.mark.parametrize("dst,wire", PAIRS)
def test_packed_equals_1d(dst, wire):
    ne0, ne1, R = 257, 9, 3
    srcs = srcs_for(1, R, ne0 * ne1, dst)
    got = oracle.reduce_2d(srcs, 2, dst, wire, ne0, ne1)
    exp = oracle.reduce(srcs, 1, dst, wire)[0]
    for g in got:
        assert_same(g, exp, dst, "packed 2-D vs 1-D")


@pytest.mark.parametrize("dst,wire", [("f32", "bf16"), ("bf16", "f16"), ("f16", "f32")])
def test_strided_rows(dst, wire):
    """Strided sources and destinations give, row by row, the packed result;
    the padding of the destinations is left untouched."""
    ne0, ne1, R = 100, 7, 4
    srcs = srcs_for(2, R, ne0 * ne1, dst)
    exp = oracle.reduce(srcs, 1, dst, wire)[0]
    s_str = [ne0 + 3 + r for r in range(R)]  # strides in elements
    d_str = [ne0 + 5, ne0]
    emb = [embed(s, ne0, st, 10 + r) for r, (s, st) in enumerate(zip(srcs, s_str))]
    outs = [embed(np.zeros(ne0 * ne1, dtype=srcs[0].dtype), ne0, st, 30 + d) for d, st in enumerate(d_str)]
    before = [o.copy() for o in outs]
    oracle.reduce_2d(emb, 2, dst, wire, ne0, ne1, src_strides=[st * ES[dst] for st in s_str],
                     dst_strides=[st * ES[dst] for st in d_str], out=outs)
    for o, b, st in zip(outs, before, d_str):
        assert_same(extract(o, ne0, ne1, st), exp, dst, "strided")
        mask = np.ones(o.size, dtype=bool)
        for j in range(ne1):
            mask[j * st: j * st + ne0] = False
        assert np.array_equal(o[mask], b[mask]), "padding written"


@pytest.mark.parametrize("dst,wire", PAIRS)
@pytest.mark.parametrize("inactive", [(0,), (1,), (0, 2), (0, 1, 2)])
def test_inactive_ranks_are_zeroed_partials(dst, wire, inactive):
    """An inactive rank behaves exactly like a rank whose tensor was zeroed."""
    R, n = 3, 4000
    srcs = srcs_for(3, R, n, dst)
    zeroed = [np.zeros_like(s) if r in inactive else s for r, s in enumerate(srcs)]
    exp = oracle.reduce(zeroed, 1, dst, wire)[0]
    holes = [None if r in inactive else s for r, s in enumerate(srcs)]
    got = oracle.reduce_2d(holes, 1, dst, wire, n, 1, inactive=inactive)[0]
    assert_same(got, exp, dst, f"inactive {inactive}")


def test_inactive_rank_is_plus_zero_not_omission():
    """-0 from every active rank plus an inactive +0 gives +0."""
    a = np.array([-0.0, -0.0], dtype=np.float32)
    got = oracle.reduce_2d([a, None], 1, "f32", "bf16", 2, 1, inactive=(1,))[0]
    assert got.view(np.uint32).tolist() == [0, 0]
    got = oracle.reduce_2d([a, a], 1, "f32", "bf16", 2, 1)[0]
    assert got.view(np.uint32).tolist() == [0x80000000, 0x80000000]


@pytest.mark.parametrize("dst", TYPES)
def test_residual_with_f32_wire_is_one_more_rank(dst):
    """With an f32 wire nothing is rounded before the sum, so adding the
    residual after the fold is the fold with the residual as the last rank."""
    R, ne0, ne1 = 3, 64, 50
    srcs = srcs_for(4, R + 1, ne0 * ne1, dst)
    got = oracle.reduce_2d(srcs[:R], 1, dst, "f32", ne0, ne1, residual=srcs[R])[0]
    exp = oracle.reduce(srcs, 1, dst, "f32")[0]
    assert_same(got, exp, dst, "residual as last rank")


@pytest.mark.parametrize("dst,wire", PAIRS)
def test_residual_matches_library_formula(dst, wire):
    R, ne0, ne1 = 2, 333, 11
    srcs = srcs_for(5, R + 1, ne0 * ne1, dst)
    got = oracle.reduce_2d(srcs[:R], 1, dst, wire, ne0, ne1, residual=srcs[R])[0]
    with np.errstate(over="ignore", invalid="ignore"):
        acc = (lib_fold_f32(srcs[:R], dst, wire) + lib_widen(dst, srcs[R])).astype(np.float32)
    assert_same(got, lib_round(dst, acc), dst, "residual")


@pytest.mark.parametrize("dst,wire", [("f32", "bf16"), ("bf16", "bf16"), ("f16", "f16")])
def test_broadcast_residual_is_tiled_row(dst, wire):
    R, ne0, ne1 = 4, 129, 13
    srcs = srcs_for(6, R, ne0 * ne1, dst)
    bias = srcs_for(7, 1, ne0, dst)[0]
    got = oracle.reduce_2d(srcs, 1, dst, wire, ne0, ne1, residual=bias, residual_stride=0)[0]
    exp = oracle.reduce_2d(srcs, 1, dst, wire, ne0, ne1, residual=np.tile(bias, ne1))[0]
    assert_same(got, exp, dst, "broadcast")


def test_residual_in_place():
    """x = x + allreduce(partials): the destination may be the residual."""
    R, n = 2, 5000
    srcs = srcs_for(8, R + 1, n, "f32")
    exp = oracle.reduce_2d(srcs[:R], 1, "f32", "bf16", n, 1, residual=srcs[R])[0]
    res = srcs[R].copy()
    oracle.reduce_2d(srcs[:R], 1, "f32", "bf16", n, 1, residual=res, out=[res])
    assert_same(res, exp, "f32", "in place")


@pytest.mark.parametrize("dst,wire", PAIRS)
def test_wire_pack_is_library_cast(dst, wire):
    (x,) = srcs_for(9, 1, 20000, dst)
    got = oracle.wire_pack(x, dst, wire)
    assert_same(got, lib_round(wire, lib_widen(dst, x)), wire, "pack")


def test_2d_rejects_null_active_source():
    with pytest.raises(ValueError):
        oracle.reduce_2d([None, np.zeros(4, np.float32)], 1, "f32", "f32", 4, 1)
