"""Reference casts taken from libraries, used to pin the oracle.

Nothing here is the oracle's code: f16 goes through numpy's float16, bf16
through torch's bfloat16, and float32 arithmetic through numpy.  Both
libraries round to nearest, ties to even, keep subnormals and overflow to
infinity (the tests check a few closed-form cases of that on their own).
"""
import numpy as np
import torch


def lib_round(name: str, x) -> np.ndarray:
    """float32 values -> storage of ``name`` (float32 or uint16 bits)."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    if name == "f32":
        return x.copy()
    if name == "f16":
        with np.errstate(over="ignore", invalid="ignore"):
            return x.astype(np.float16).view(np.uint16)
    if name == "bf16":
        t = torch.from_numpy(x).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise KeyError(name)


def lib_widen(name: str, bits) -> np.ndarray:
    """storage of ``name`` -> exact float32 values."""
    bits = np.ascontiguousarray(bits).ravel()
    if name == "f32":
        return bits.view(np.float32).copy()
    if name == "f16":
        return bits.view(np.float16).astype(np.float32)
    if name == "bf16":
        t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
        return t.to(torch.float32).numpy()
    raise KeyError(name)


def lib_reduce(srcs, dst: str, wire: str) -> np.ndarray:
    """The reduction written with library casts and numpy float32 adds."""
    acc = None
    for s in srcs:
        w = lib_widen(wire, lib_round(wire, lib_widen(dst, s)))
        if acc is None:
            acc = w.copy()
        else:
            with np.errstate(over="ignore", invalid="ignore"):
                acc = (acc + w).astype(np.float32)
    return lib_round(dst, acc)


def as_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a).ravel()
    return a.view(np.uint32) if a.dtype.itemsize == 4 else a.view(np.uint16)


def is_nan_bits(bits: np.ndarray, name: str) -> np.ndarray:
    if name == "f32":
        return ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x007FFFFF) != 0)
    if name == "f16":
        return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x03FF) != 0)
    if name == "bf16":
        return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)
    raise KeyError(name)


def mismatches(a, b, name: str) -> np.ndarray:
    """Indices where a and b differ bitwise, any NaN matching any NaN."""
    ab, bb = as_bits(a), as_bits(b)
    na, nb = is_nan_bits(ab, name), is_nan_bits(bb, name)
    bad = (ab != bb) & ~(na & nb)
    return np.nonzero(bad)[0]


def assert_same(a, b, name: str, what: str = ""):
    ab, bb = as_bits(a), as_bits(b)
    if ab.shape != bb.shape:
        raise AssertionError(f"{what}: {ab.size} elements against {bb.size}")
    if np.array_equal(ab, bb):  # the common case, without the NaN masks' temporaries
        return
    bad = mismatches(a, b, name)
    if bad.size:
        i = int(bad[0])
        ab, bb = as_bits(a), as_bits(b)
        raise AssertionError(
            f"{what}: {bad.size} of {ab.size} elements differ; first at {i}: "
            f"{int(ab[i]):#x} vs {int(bb[i]):#x}")
