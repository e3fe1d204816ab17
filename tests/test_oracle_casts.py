"""Pins for the oracle's casts (CPU only).

The oracle rounds by the textbook definition (scale to the grid, pick the
nearer integer, ties to even).  These tests tie it to three things that are
not that code: hand-derived closed forms, library conversions (numpy float16,
torch bfloat16), and a brute-force search for the nearest value among every
finite value of the target format.
"""
import os
import threading

import numpy as np
import pytest

import oracle
from tests.libcasts import assert_same, lib_round, lib_widen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "cast_closed_forms.txt")


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, name, inp, exp = line.split()[:4]
            rows.append((kind, name, int(inp, 16), int(exp, 16), line))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: f"{r[0]}-{r[1]}-{r[2]:#x}")
def test_closed_form(row):
    kind, name, inp, exp, line = row
    L = oracle.lib()
    code = oracle.DTYPES[name]
    if kind == "round":
        x = np.array([inp], dtype=np.uint32).view(np.float32)[0]
        got = L.orc_round(code, float(x))
        assert got == exp, f"{line}: got {got:#x}"
        # the libraries agree with the hand derivation as well
        lib = int(lib_round(name, np.array([x], dtype=np.float32))[0])
        assert lib == exp, f"{line}: library gives {lib:#x}"
    else:
        got = np.float32(L.orc_widen(code, inp)).view(np.uint32)
        assert int(got) == exp, f"{line}: got {int(got):#x}"


def _structured_inputs(name: str) -> np.ndarray:
    """Every sign/exponent/kept-fraction combination crossed with the
    rounding-bit patterns that decide a tie (0, 1, just below half, half,
    just above half, all ones) and a few random ones; plus random float32
    patterns across the target's subnormal range, where the rounding
    position moves."""
    rng = np.random.Generator(np.random.PCG64(12345))
    if name == "bf16":
        drop = 16
    else:
        drop = 13
    half = 1 << (drop - 1)
    low = np.array([0, 1, half - 1, half, half + 1, (1 << drop) - 1], dtype=np.uint64)
    low = np.concatenate([low, rng.integers(0, 1 << drop, 10, dtype=np.uint64)])
    high = np.arange(0, 1 << (32 - drop), dtype=np.uint64) << np.uint64(drop)
    x = (high[:, None] | low[None, :]).ravel().astype(np.uint32)
    if name == "f16":
        # float32 exponents 101..113 cover binary16's subnormal range and the
        # first normal binade; draw random fractions there
        e = rng.integers(101, 114, 1 << 22, dtype=np.uint32)
        s = rng.integers(0, 2, 1 << 22, dtype=np.uint32)
        m = rng.integers(0, 1 << 23, 1 << 22, dtype=np.uint32)
        x = np.concatenate([x, (s << 31) | (e << 23) | m])
    else:
        # float32 subnormals and the first normal binade
        e = rng.integers(0, 2, 1 << 21, dtype=np.uint32)
        s = rng.integers(0, 2, 1 << 21, dtype=np.uint32)
        m = rng.integers(0, 1 << 23, 1 << 21, dtype=np.uint32)
        x = np.concatenate([x, (s << 31) | (e << 23) | m])
    return x.view(np.float32)


@pytest.mark.parametrize("name", ["f16", "bf16"])
def test_round_matches_library(name):
    x = _structured_inputs(name)
    assert_same(oracle.round_to(name, x), lib_round(name, x), name, f"round {name} vs library")


def _all_finite_values(name: str):
    """Sorted non-negative finite values of the format (float64) with their
    bit patterns, followed by the first power of two past the largest finite
    value, which stands for overflow (its pattern is +inf's)."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = lib_widen(name, bits).astype(np.float64)
    keep = np.isfinite(vals) & (np.signbit(vals) == 0)
    vals, bits = vals[keep], bits[keep]
    order = np.argsort(vals, kind="stable")
    vals, bits = vals[order], bits[order]
    inf_bits = np.uint16(0x7C00 if name == "f16" else 0x7F80)
    top = 2.0 ** (16 if name == "f16" else 128)
    return np.append(vals, top), np.append(bits, inf_bits)


@pytest.mark.parametrize("name", ["f16", "bf16"])
def test_round_is_nearest_value(name):
    """Brute force: the nearest of all the format's values, ties to the even
    bit pattern, overflow where the nearest is the power past the top."""
    x = _structured_inputs(name)
    x = x[np.isfinite(x)]
    vals, bits = _all_finite_values(name)
    a = np.abs(x.astype(np.float64))
    hi = np.clip(np.searchsorted(vals, a, side="left"), 1, vals.size - 1)
    lo = hi - 1
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((bits[hi] & 1) == 0))
    pick_hi |= a >= vals[-1]
    exp = np.where(pick_hi, bits[hi], bits[lo]).astype(np.uint16)
    exp |= np.where(np.signbit(x), np.uint16(0x8000), np.uint16(0))
    assert_same(oracle.round_to(name, x), exp, name, f"round {name} vs nearest value")


@pytest.mark.parametrize("name", ["f16", "bf16"])
def test_widen_exhaustive(name):
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    assert_same(oracle.widen(name, bits), lib_widen(name, bits), "f32", f"widen {name}")
    # round-trip identity on every pattern (NaN as a class)
    assert_same(oracle.round_to(name, oracle.widen(name, bits)), bits, name, f"{name} round-trip")


def test_f32_is_identity():
    rng = np.random.Generator(np.random.PCG64(7))
    x = rng.integers(0, 1 << 32, 1 << 16, dtype=np.uint64).astype(np.uint32).view(np.float32)
    assert_same(oracle.round_to("f32", x), x, "f32", "f32 round")
    assert_same(oracle.widen("f32", x), x, "f32", "f32 widen")


@pytest.mark.exhaustive
@pytest.mark.parametrize("name", ["f16", "bf16"])
def test_round_exhaustive(name):
    """Every float32 bit pattern against the library conversion."""
    chunk = 1 << 24
    errors = []

    def run(starts):
        for s in starts:
            x = np.arange(s, s + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
            try:
                assert_same(oracle.round_to(name, x), lib_round(name, x), name, f"chunk {s:#x}")
            except AssertionError as e:  # pragma: no cover - reported below
                errors.append(str(e))

    starts = list(range(0, 1 << 32, chunk))
    n = os.cpu_count() or 4
    threads = [threading.Thread(target=run, args=(starts[i::n],)) for i in range(n)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:3]
