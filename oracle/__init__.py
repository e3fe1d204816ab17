"""Python access to the scalar CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The product library
never loads it, and it never loads the product library.

Arrays are numpy arrays in storage form: ``f32`` as ``float32``; ``f16`` and
``bf16`` as ``uint16`` bit patterns (a ``float16`` array is accepted for
``f16`` and viewed as its bits).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
_STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16}
CFLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]

_lock = threading.Lock()
_default = None


def _stale() -> bool:
    if not os.path.exists(_LIB_PATH):
        return True
    t = os.path.getmtime(_LIB_PATH)
    return any(os.path.getmtime(p) > t for p in (_SRC, _HDR))


def compile_to(src: str, out: str) -> str:
    """Compile an oracle source file into a shared library (atomic rename)."""
    d = os.path.dirname(os.path.abspath(out))
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=d)
    os.close(fd)
    try:
        subprocess.run(["gcc", *CFLAGS, "-I", _HERE, "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source with gcc."""
    if force or _stale():
        compile_to(_SRC, _LIB_PATH)
    return _LIB_PATH


def storage_dtype(name: str):
    return _STORAGE[name]


def _as_storage(a: np.ndarray, name: str) -> np.ndarray:
    a = np.ascontiguousarray(a)
    want = _STORAGE[name]
    if a.dtype == want:
        return a
    if a.dtype.itemsize == np.dtype(want).itemsize:
        return a.view(want)
    raise TypeError(f"array of {a.dtype} is not {name} storage")


def _ptr_array(arrays):
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


class Oracle:
    """One loaded copy of the oracle library."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        L.orc_elem_size.argtypes = [i]
        L.orc_elem_size.restype = sz
        L.orc_widen.argtypes = [i, ctypes.c_uint32]
        L.orc_widen.restype = ctypes.c_float
        L.orc_round.argtypes = [i, ctypes.c_float]
        L.orc_round.restype = ctypes.c_uint32
        L.orc_widen_array.argtypes = [i, vp, vp, sz]
        L.orc_widen_array.restype = None
        L.orc_round_array.argtypes = [i, vp, vp, sz]
        L.orc_round_array.restype = None
        L.orc_reduce_range.argtypes = [i, vp, vp, i, sz, sz, i, i]
        L.orc_reduce_range.restype = i
        L.orc_reduce.argtypes = [i, vp, vp, i, sz, i, i]
        L.orc_reduce.restype = i
        ll_p = ctypes.POINTER(ctypes.c_longlong)
        L.orc_reduce_2d.argtypes = [i, vp, ll_p, ctypes.c_uint, vp, ctypes.c_longlong, vp, ll_p, i, sz, sz, i, i]
        L.orc_reduce_2d.restype = i
        L.orc_wire_pack.argtypes = [vp, vp, sz, i, i]
        L.orc_wire_pack.restype = i
        self.lib = L
        self.path = path

    def widen(self, name: str, bits: np.ndarray) -> np.ndarray:
        """Exact float32 value of each stored element."""
        bits = _as_storage(bits, name).ravel()
        out = np.empty(bits.size, dtype=np.float32)
        self.lib.orc_widen_array(DTYPES[name], bits.ctypes.data, out.ctypes.data, bits.size)
        return out

    def round_to(self, name: str, x: np.ndarray) -> np.ndarray:
        """Round-to-nearest-even cast of float32 values, in storage form."""
        x = np.ascontiguousarray(x, dtype=np.float32).ravel()
        out = np.empty(x.size, dtype=_STORAGE[name])
        self.lib.orc_round_array(DTYPES[name], x.ctypes.data, out.ctypes.data, x.size)
        return out

    def reduce(self, srcs, n_dsts: int, dst_dtype: str, wire_dtype: str,
               begin: int = 0, end: int | None = None, out=None):
        """Reduce R source arrays (storage form of ``dst_dtype``) into
        ``n_dsts`` new arrays (or into ``out``), over ``[begin, end)``."""
        srcs = [_as_storage(s, dst_dtype).ravel() for s in srcs]
        nelem = srcs[0].size
        if any(s.size != nelem for s in srcs):
            raise ValueError("source arrays differ in length")
        if end is None:
            end = nelem
        if out is None:
            out = [np.zeros(nelem, dtype=_STORAGE[dst_dtype]) for _ in range(n_dsts)]
        else:
            out = [_as_storage(o, dst_dtype).reshape(-1) for o in out]
        if len(out) != n_dsts:
            raise ValueError("need one output array per destination")
        rc = self.lib.orc_reduce_range(len(srcs), _ptr_array(srcs), _ptr_array(out), n_dsts,
                                       begin, end, DTYPES[dst_dtype], DTYPES[wire_dtype])
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return out


    def reduce_2d(self, srcs, n_dsts, dst_dtype, wire_dtype, ne0, ne1, src_strides=None, dst_strides=None,
                  inactive=(), residual=None, residual_stride=None, out=None):
        """2-D reduction with row strides (bytes), inactive ranks (+0
        operands; their source may be None), and an optional residual
        (``residual_stride`` 0 = one row broadcast to every row).  Sources
        and outputs are flat storage arrays holding the strided rows."""
        es = 4 if dst_dtype == "f32" else 2
        srcs = [None if s is None else _as_storage(s, dst_dtype).ravel() for s in srcs]
        mask = 0
        for r in inactive:
            mask |= 1 << r
        if out is None:
            ds = dst_strides or [ne0 * es] * n_dsts
            out = [np.zeros(max(1, ((ne1 - 1) * ds[d] + ne0 * es) // es) if ne1 else 1, dtype=_STORAGE[dst_dtype])
                   for d in range(n_dsts)]
        else:
            out = [_as_storage(o, dst_dtype).reshape(-1) for o in out]
        src_arr = (ctypes.c_void_p * len(srcs))(*[None if s is None else s.ctypes.data for s in srcs])
        ll = ctypes.c_longlong
        ss = None if src_strides is None else (ll * len(src_strides))(*src_strides)
        dd = None if dst_strides is None else (ll * len(dst_strides))(*dst_strides)
        res = None
        if residual is not None:
            residual = _as_storage(residual, dst_dtype).ravel()
            res = residual.ctypes.data
            if residual_stride is None:
                residual_stride = ne0 * es
        rc = self.lib.orc_reduce_2d(len(srcs), src_arr, ss, mask, res, residual_stride or 0, _ptr_array(out), dd,
                                    n_dsts, ne0, ne1, DTYPES[dst_dtype], DTYPES[wire_dtype])
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return out

    def wire_pack(self, src, dst_dtype, wire_dtype):
        src = _as_storage(src, dst_dtype).ravel()
        out = np.empty(src.size, dtype=_STORAGE[wire_dtype])
        if self.lib.orc_wire_pack(src.ctypes.data, out.ctypes.data, src.size, DTYPES[dst_dtype],
                                  DTYPES[wire_dtype]) != 0:
            raise ValueError("oracle rejected the arguments")
        return out


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def lib() -> ctypes.CDLL:
    return default().lib


def widen(name, bits):
    return default().widen(name, bits)


def round_to(name, x):
    return default().round_to(name, x)


def reduce(srcs, n_dsts, dst_dtype, wire_dtype, begin=0, end=None, out=None):
    return default().reduce(srcs, n_dsts, dst_dtype, wire_dtype, begin, end, out)


def reduce_2d(*args, **kwargs):
    return default().reduce_2d(*args, **kwargs)


def wire_pack(src, dst_dtype, wire_dtype):
    return default().wire_pack(src, dst_dtype, wire_dtype)
