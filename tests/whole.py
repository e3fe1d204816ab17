"""The oracle over whole full-size tensors, on every host core.

Every output element depends only on the same element of the inputs, so the
oracle can run over contiguous ranges (of elements, or of whole rows for the
2-D layouts) in parallel threads and write into one output array: the bytes
are exactly those of a single serial pass.  The oracle's C calls release the
GIL, so the threads run at once."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _split(n: int, parts: int):
    parts = max(1, min(parts, n))
    return [(n * k // parts, n * (k + 1) // parts) for k in range(parts)]


def _run(fn, ranges):
    with ThreadPoolExecutor(len(ranges)) as pool:
        list(pool.map(lambda r: fn(*r), ranges))


def reduce(srcs, dst: str, wire: str) -> np.ndarray:
    """oracle.reduce over every element (one destination)."""
    n = srcs[0].size
    out = np.empty(n, dtype=oracle.storage_dtype(dst))
    _run(lambda a, b: oracle.reduce(srcs, 1, dst, wire, begin=a, end=b, out=[out]), _split(n, 4 * host_threads()))
    return out


def wire_pack(src, dst: str, wire: str) -> np.ndarray:
    """oracle.wire_pack over every element."""
    n = src.size
    out = np.empty(n, dtype=oracle.storage_dtype(wire))

    def part(a, b):
        out[a:b] = oracle.wire_pack(src[a:b], dst, wire)

    _run(part, _split(n, 4 * host_threads()))
    return out


def reduce_rows(srcs, dst: str, wire: str, ne0: int, ne1: int, inactive=(), residual=None,
                residual_kind: str = "") -> np.ndarray:
    """oracle.reduce_2d over all ne1 packed rows of ne0 elements, with
    inactive ranks (None sources), and a residual that is a full tensor
    (``residual_kind`` "full") or one bias row ("row")."""
    out = np.empty(ne0 * ne1, dtype=oracle.storage_dtype(dst))

    def part(r0, r1):
        a, b = r0 * ne0, r1 * ne0
        res, res_stride = None, None
        if residual_kind == "full":
            res = residual[a:b]
        elif residual_kind == "row":
            res, res_stride = residual, 0
        holes = [None if r in inactive else s[a:b] for r, s in enumerate(srcs)]
        oracle.reduce_2d(holes, 1, dst, wire, ne0, r1 - r0, inactive=inactive, residual=res,
                         residual_stride=res_stride, out=[out[a:b]])

    _run(part, _split(ne1, 4 * host_threads()))
    return out
