"""Pins for the oracle's reduction (CPU only).

What the pages and the arithmetic fix, checked against the oracle:
  * R = 1 is the wire round-trip of the single operand;
  * R = 2 is symmetric, so both ranks get the same bits
    (ggml-cuda allreduce.cu, ggml_cuda_ar_kernel "Phase 3": each side rounds
    its own value through the wire type exactly as the peer's value was
    rounded, which is what makes the two results equal);
  * small integers exact in the wire type sum to the exact integer;
  * the fold is left to right in rank order (ggml-hexagon allreduce-ops.c,
    DEFINE_ALLREDUCE_THREAD_DMA_1D: s0 + s1, then + s2 ...), shown by a
    constructed case whose result depends on the order;
  * every destination receives the same bits;
  * splitting the element range into chunks changes nothing
    (allreduce.cu, ggml_cuda_ar_allreduce_copy_outer and the chunk loop of
    ggml_cuda_ar_allreduce);
  * the whole reduction equals the same formula evaluated with library casts
    and numpy float32 adds, on inputs full of edge values.
"""
import itertools

import numpy as np
import pytest

import oracle
from tests.libcasts import assert_same, lib_reduce, lib_round, lib_widen

TYPES = ["f32", "f16", "bf16"]
PAIRS = list(itertools.product(TYPES, TYPES))  # (dst, wire)


def edgy_f32(rng, n):
    """float32 values mixing normals with edge cases of every format."""
    x = rng.standard_normal(n).astype(np.float32)
    kind = rng.integers(0, 10, n)
    sign = np.where(rng.integers(0, 2, n) == 1, -1.0, 1.0).astype(np.float32)
    big = rng.uniform(5.4e4, 6.6e4, n).astype(np.float32) * sign
    tiny = np.exp(rng.uniform(np.log(1e-7), np.log(6e-5), n)).astype(np.float32) * sign
    sub32 = (rng.integers(1, 1 << 23, n).astype(np.uint32)).view(np.float32) * sign
    special = np.array([0.0, -0.0, 65504.0, 65520.0, -65520.0, 2.0 ** -24, 2.0 ** -25,
                        np.inf, -np.inf, np.nan, 3.0e38, -3.0e38, 1.0 + 2.0 ** -8,
                        1.0 + 2.0 ** -11], dtype=np.float32)
    pick = special[rng.integers(0, special.size, n)]
    x = np.where(kind == 1, big, x)
    x = np.where(kind == 2, tiny, x)
    x = np.where(kind == 3, sub32, x)
    x = np.where(kind == 4, pick, x)
    with np.errstate(over="ignore"):
        x = np.where(kind == 5, x * np.float32(1e4), x)
    return x.astype(np.float32)


def make_srcs(rng, R, n, dst):
    return [lib_round(dst, edgy_f32(rng, n)) for _ in range(R)]


@pytest.mark.parametrize("dst,wire", PAIRS)
def test_r1_is_wire_round_trip(dst, wire):
    rng = np.random.Generator(np.random.PCG64(1))
    (x,) = make_srcs(rng, 1, 20000, dst)
    got = oracle.reduce([x], 1, dst, wire)[0]
    exp = lib_round(dst, lib_widen(wire, lib_round(wire, lib_widen(dst, x))))
    assert_same(got, exp, dst, f"R=1 {dst}/{wire}")


@pytest.mark.parametrize("dst,wire", PAIRS)
def test_r2_symmetric(dst, wire):
    rng = np.random.Generator(np.random.PCG64(2))
    a, b = make_srcs(rng, 2, 20000, dst)
    ab = oracle.reduce([a, b], 1, dst, wire)[0]
    ba = oracle.reduce([b, a], 1, dst, wire)[0]
    assert_same(ab, ba, dst, f"R=2 symmetry {dst}/{wire}")


@pytest.mark.parametrize("dst,wire", PAIRS)
@pytest.mark.parametrize("R", [1, 2, 3, 5, 8, 16])
def test_matches_library_formula(dst, wire, R):
    rng = np.random.Generator(np.random.PCG64(100 + R))
    srcs = make_srcs(rng, R, 6000, dst)
    got = oracle.reduce(srcs, 1, dst, wire)[0]
    assert_same(got, lib_reduce(srcs, dst, wire), dst, f"R={R} {dst}/{wire}")


@pytest.mark.parametrize("wire,limit", [("bf16", 256), ("f16", 2048), ("f32", 1 << 20)])
@pytest.mark.parametrize("R", [2, 4, 16])
def test_exact_integer_sums(wire, limit, R):
    """|v| <= 2^p is exact in a format of precision p, so the wire cast is
    exact, and the float sum of at most 16 such values is exact too."""
    rng = np.random.Generator(np.random.PCG64(R))
    ints = rng.integers(-limit, limit + 1, (R, 5000))
    srcs = [v.astype(np.float32) for v in ints]
    got = oracle.reduce(srcs, 1, "f32", wire)[0]
    assert np.array_equal(got, ints.sum(axis=0).astype(np.float32))


def test_exact_integer_sums_bf16_dst():
    """bf16 destination: |sum| <= 128 is exact in bfloat16."""
    rng = np.random.Generator(np.random.PCG64(9))
    ints = rng.integers(-8, 9, (16, 5000))
    srcs = [lib_round("bf16", v.astype(np.float32)) for v in ints]
    got = oracle.widen("bf16", oracle.reduce(srcs, 1, "bf16", "bf16")[0])
    assert np.array_equal(got, ints.sum(axis=0).astype(np.float32))


def test_rank_order_matters_and_is_ascending():
    """In float, (1e8 + 1) - 1e8 is 0 (1e8 + 1 rounds back to 1e8) while
    (1e8 - 1e8) + 1 is 1: the result shows which order the fold used."""
    one = [np.array([v], dtype=np.float32) for v in (1e8, 1.0, -1e8)]
    assert oracle.reduce(one, 1, "f32", "f32")[0][0] == 0.0
    two = [np.array([v], dtype=np.float32) for v in (1e8, -1e8, 1.0)]
    assert oracle.reduce(two, 1, "f32", "f32")[0][0] == 1.0


def test_signed_zero_and_specials():
    f = lambda *v: [np.array([x], dtype=np.float32) for x in v]  # noqa: E731
    bits = lambda a: int(a.view(np.uint32)[0])  # noqa: E731
    # the fold starts from the first operand: a lone -0 stays -0
    assert bits(oracle.reduce(f(-0.0), 1, "f32", "bf16")[0]) == 0x80000000
    assert bits(oracle.reduce(f(-0.0, -0.0), 1, "f32", "f16")[0]) == 0x80000000
    assert bits(oracle.reduce(f(-0.0, 0.0), 1, "f32", "f16")[0]) == 0x00000000
    # a wire overflow becomes inf; opposite infinities give NaN
    assert oracle.reduce(f(65520.0, 1.0), 1, "f32", "f16")[0][0] == np.inf
    assert np.isnan(oracle.reduce(f(65520.0, -65520.0), 1, "f32", "f16")[0][0])
    # an f16 subnormal operand survives the wire: 2^-24 + 2^-24 = 2^-23
    assert oracle.reduce(f(2.0 ** -24, 2.0 ** -24), 1, "f32", "f16")[0][0] == 2.0 ** -23
    # a float sum can overflow on its own
    assert oracle.reduce(f(3e38, 3e38), 1, "f32", "f32")[0][0] == np.inf
    # a bf16 result overflows when the float sum passes bf16's top midpoint
    top = np.array([0x7F7F0000], dtype=np.uint32).view(np.float32)[0]
    tb = lib_round("bf16", np.array([top], dtype=np.float32))
    r = oracle.reduce([tb, tb], 1, "bf16", "f32")[0]
    assert int(r[0]) == 0x7F80


@pytest.mark.parametrize("n_dsts", [1, 2, 7, 16])
def test_every_destination_identical(n_dsts):
    rng = np.random.Generator(np.random.PCG64(n_dsts))
    srcs = make_srcs(rng, 4, 3000, "f32")
    outs = oracle.reduce(srcs, n_dsts, "f32", "f16")
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


@pytest.mark.parametrize("dst,wire", [("f32", "bf16"), ("bf16", "bf16"), ("f32", "f16")])
def test_chunking_is_invisible(dst, wire):
    rng = np.random.Generator(np.random.PCG64(33))
    E = 3 * 4099 + 5
    srcs = make_srcs(rng, 3, E, dst)
    whole = oracle.reduce(srcs, 1, dst, wire)[0]
    for c in (1, 3, 4099, E):
        out = [np.zeros_like(whole)]
        for b in range(0, E, c):
            oracle.reduce(srcs, 1, dst, wire, begin=b, end=min(E, b + c), out=out)
        assert_same(out[0], whole, dst, f"chunk {c}")


def test_in_place_destination():
    """The reference reduces in place (send and receive buffers are the same
    tensor); writing into a source gives the same bits."""
    rng = np.random.Generator(np.random.PCG64(44))
    srcs = make_srcs(rng, 3, 5000, "f32")
    exp = oracle.reduce(srcs, 1, "f32", "bf16")[0]
    srcs2 = [s.copy() for s in srcs]
    oracle.reduce(srcs2, 1, "f32", "bf16", out=[srcs2[1]])
    assert_same(srcs2[1], exp, "f32", "in place")


def test_rejects_bad_arguments():
    L = oracle.lib()
    assert L.orc_reduce(0, None, None, 1, 1, 0, 0) == -1
    x = np.zeros(4, dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.reduce([x], 1, "f32", "f32", out=[x, x])
