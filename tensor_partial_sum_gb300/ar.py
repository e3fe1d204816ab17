"""ctypes binding of libtps_ar.so, one Python function per C entry point.

Argument marshalling only: tensors become device pointers, Python lists
become pointer arrays, torch streams become ``cudaStream_t`` handles, and a
non-zero status becomes an ``ARError``.  Every step of the reduction runs in
the library's CUDA kernels; there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import struct

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libtps_ar.so")

AR_F32, AR_F16, AR_BF16 = 0, 1, 2
DTYPE_CODES = {"f32": AR_F32, "f16": AR_F16, "bf16": AR_BF16}

AR_OK = 0
STATUS_NAMES = {0: "AR_OK", 1: "AR_ERR_INVALID_ARG", 2: "AR_ERR_UNSUPPORTED", 3: "AR_ERR_TOO_LARGE",
                4: "AR_ERR_NOT_INITIALIZED", 5: "AR_ERR_OVERLAP", 6: "AR_ERR_CUDA"}
VARIANTS = {"auto": 0, "naive": 1, "latency": 2, "bandwidth": 3, "scalar": 4, "tma": 5}
KEYS = {"ranks": 0, "max_elems": 1, "device": 2, "sm_count": 3, "latency_max_bytes": 4,
        "forced_variant": 5, "last_variant": 6, "fault_inject": 7, "bw_blocks_per_sm": 8,
        "host_chunk_bytes": 9, "device_status": 10, "tma_drop_tile": 11}

_lib = None


class ArLayout(ctypes.Structure):
    """ar_layout of include/ar.h."""
    _fields_ = [("ne0", ctypes.c_size_t), ("ne1", ctypes.c_size_t),
                ("src_row_bytes", ctypes.POINTER(ctypes.c_int64)),
                ("dst_row_bytes", ctypes.POINTER(ctypes.c_int64)),
                ("residual", ctypes.c_void_p), ("residual_row_bytes", ctypes.c_int64),
                ("inactive_mask", ctypes.c_uint32)]


class ARError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {STATUS_NAMES.get(status, status)} ({ar_status_string(status)})")


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is not built: run `python -m tensor_partial_sum_gb300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        vp, sz, i, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64
        # pointer arrays travel as packed bytes (see _ptrs): the C side reads
        # R or n_dsts 64-bit addresses from the buffer
        pp = ctypes.c_char_p
        L.ar_init.argtypes = [i, sz]
        L.ar_init.restype = i
        L.ar_reduce.argtypes = [pp, pp, i, sz, i, i, vp]
        L.ar_reduce.restype = i
        L.ar_free.argtypes = []
        L.ar_free.restype = None
        L.ar_status_string.argtypes = [i]
        L.ar_status_string.restype = ctypes.c_char_p
        L.ar_check_args.argtypes = [i, pp, pp, i, sz, sz, i, i]
        L.ar_check_args.restype = i
        L.ar_reduce_variant.argtypes = [pp, pp, i, sz, i, i, i, i, vp]
        L.ar_reduce_variant.restype = i
        L.ar_query.argtypes = [i, ctypes.POINTER(i64)]
        L.ar_query.restype = i
        L.ar_set_option.argtypes = [i, i64]
        L.ar_set_option.restype = i
        L.ar_reduce_host.argtypes = [pp, pp, i, sz, i, i, pp, pp, vp]
        L.ar_reduce_host.restype = i
        lp = ctypes.POINTER(ArLayout)
        L.ar_reduce_ex.argtypes = [pp, pp, i, lp, i, i, vp]
        L.ar_reduce_ex.restype = i
        L.ar_check_layout.argtypes = [i, pp, pp, i, lp, sz, i, i]
        L.ar_check_layout.restype = i
        L.ar_wire_pack.argtypes = [vp, vp, sz, i, i, vp]
        L.ar_wire_pack.restype = i
        L.ar_reduce_host_noalloc.argtypes = [pp, pp, i, sz, i, i, vp]
        L.ar_reduce_host_noalloc.restype = i
        _lib = L
    return _lib


# ---- marshalling helpers -------------------------------------------------

def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):  # numpy array (host buffers)
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x).__name__}")


AR_MAX_RANKS = 16


_PTR_ARRAY = struct.Struct(f"={AR_MAX_RANKS}Q")


def _ptrs(xs):
    """Pointer array (packed native 64-bit addresses, 0 for None) padded to
    at least AR_MAX_RANKS entries, so a list shorter than the context's R is
    rejected (NULL source) instead of being read past its end.  Packing with
    struct costs a fraction of building a ctypes array of c_void_p."""
    if xs is None:
        return None
    ptrs = [_ptr(x) or 0 for x in xs]
    if len(ptrs) <= AR_MAX_RANKS:
        return _PTR_ARRAY.pack(*ptrs, *([0] * (AR_MAX_RANKS - len(ptrs))))
    return struct.pack(f"={len(ptrs)}Q", *ptrs)


ESIZE = {AR_F32: 4, AR_F16: 2, AR_BF16: 2}


def _checked(xs, nelem, dcode, where, call):
    """Check the buffers of a 1-D call before their addresses reach the
    library: torch tensors and numpy arrays must be contiguous, hold at
    least ``nelem`` elements of the call's type, and live where the entry
    point reads them (``where`` = "device" or "host").  Plain integers are
    addresses the caller vouches for.  A wrong buffer would otherwise be
    read or written past its end by a kernel."""
    if xs is None:
        return xs
    need = nelem * ESIZE.get(dcode, 1)
    for k, x in enumerate(xs):
        if x is None or isinstance(x, int):
            continue
        if hasattr(x, "data_ptr"):
            if (x.device.type == "cuda") != (where == "device"):
                raise TypeError(f"{call}: buffer {k} is a {x.device.type} tensor, a {where} buffer is needed")
            if not x.is_contiguous():
                raise ValueError(f"{call}: buffer {k} is not contiguous")
            have = x.numel() * x.element_size()
        elif hasattr(x, "ctypes"):
            if where != "host":
                raise TypeError(f"{call}: buffer {k} is a numpy array, a device buffer is needed")
            if not x.flags["C_CONTIGUOUS"]:
                raise ValueError(f"{call}: buffer {k} is not contiguous")
            have = x.nbytes
        else:
            continue
        if have < need:
            raise ValueError(f"{call}: buffer {k} holds {have} bytes, the call needs {need}")
    return xs


def _reach(x) -> int | None:
    """Bytes a kernel may touch from a CUDA tensor's first element to the end
    of its storage (None for raw addresses); a non-CUDA tensor is refused."""
    if x is None or isinstance(x, int) or not hasattr(x, "data_ptr"):
        return None
    if x.device.type != "cuda":
        raise TypeError(f"a {x.device.type} tensor where a device buffer is needed")
    st = x.untyped_storage()
    return st.data_ptr() + st.nbytes() - x.data_ptr()


def _dtype_code(d) -> int:
    if isinstance(d, int):
        return d
    if isinstance(d, str):
        return DTYPE_CODES[d]
    import torch
    return {torch.float32: AR_F32, torch.float16: AR_F16, torch.bfloat16: AR_BF16}[d]


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _infer(srcs, nelem, dst_dtype):
    """nelem and dtype code from the first buffer unless given: torch tensors
    and numpy arrays (float32 -> f32, float16 -> f16; uint16 bit patterns are
    ambiguous between f16 and bf16 and need an explicit dst_dtype)."""
    t = srcs[0] if srcs else None
    if nelem is None:
        nelem = t.numel() if hasattr(t, "numel") else int(t.size)
    if dst_dtype is None:
        if hasattr(t, "numel"):
            dst_dtype = t.dtype
        else:
            name = {"float32": "f32", "float16": "f16"}.get(str(t.dtype))
            if name is None:
                raise TypeError(f"cannot tell the element type of a {t.dtype} array: pass dst_dtype")
            dst_dtype = name
    return nelem, _dtype_code(dst_dtype)


def _check(status: int, call: str) -> int:
    if status != AR_OK:
        raise ARError(status, call)
    return status


# ---- entry points ----------------------------------------------------------

def ar_status_string(status: int) -> str:
    return lib().ar_status_string(status).decode()


def ar_init(R: int, max_elems: int) -> None:
    _check(lib().ar_init(R, max_elems), "ar_init")


def ar_free() -> None:
    lib().ar_free()


def ar_reduce(srcs, dsts, nelem=None, dst_dtype=None, wire_dtype="bf16", stream=None) -> None:
    """Enqueue one reduction of ``srcs`` (R tensors or device pointers) into
    every tensor of ``dsts``.  ``nelem``/``dst_dtype`` default to the first
    source tensor's; ``stream`` defaults to torch's current stream."""
    nelem, dcode = _infer(srcs, nelem, dst_dtype)
    _checked(srcs, nelem, dcode, "device", "ar_reduce")
    _checked(dsts, nelem, dcode, "device", "ar_reduce")
    _check(lib().ar_reduce(_ptrs(srcs), _ptrs(dsts), len(dsts), nelem, dcode, _dtype_code(wire_dtype),
                           _stream(stream)), "ar_reduce")


def ar_reduce_variant(srcs, dsts, variant="auto", grid_blocks=0, nelem=None, dst_dtype=None,
                      wire_dtype="bf16", stream=None) -> None:
    nelem, dcode = _infer(srcs, nelem, dst_dtype)
    _checked(srcs, nelem, dcode, "device", "ar_reduce_variant")
    _checked(dsts, nelem, dcode, "device", "ar_reduce_variant")
    v = VARIANTS[variant] if isinstance(variant, str) else variant
    _check(lib().ar_reduce_variant(_ptrs(srcs), _ptrs(dsts), len(dsts), nelem, dcode, _dtype_code(wire_dtype),
                                   v, grid_blocks, _stream(stream)), "ar_reduce_variant")


class PreparedReduce:
    """One ar_reduce_variant call with its arguments fixed: the buffer
    checks and the pointer arrays are done once, so each call is a single
    C call (for eager code that repeats the same reduction, e.g. every
    decode step; a CUDA graph removes the per-call cost altogether).  Holds
    references to the buffers it was given."""

    def __init__(self, srcs, dsts, nelem=None, dst_dtype=None, wire_dtype="bf16", variant="auto", stream=None):
        nelem, dcode = _infer(srcs, nelem, dst_dtype)
        _checked(srcs, nelem, dcode, "device", "PreparedReduce")
        _checked(dsts, nelem, dcode, "device", "PreparedReduce")
        self._keep = (list(srcs), list(dsts))
        self._args = (_ptrs(srcs), _ptrs(dsts), len(dsts), nelem, dcode, _dtype_code(wire_dtype),
                      VARIANTS[variant] if isinstance(variant, str) else variant, 0)
        self._stream = None if stream is None else _stream(stream)
        self._fn = lib().ar_reduce_variant

    def __call__(self, stream=None):
        """Enqueue the reduction on ``stream`` (default: the one given at
        preparation, else torch's current stream)."""
        s = _stream(stream) if stream is not None else (self._stream if self._stream is not None else _stream(None))
        st = self._fn(*self._args, s)
        if st != AR_OK:
            raise ARError(st, "ar_reduce")


def ar_check_args(R, srcs, dsts, n_dsts, nelem, max_elems, dst_dtype, wire_dtype) -> int:
    """Host-only validation; returns the status code (does not raise)."""
    return lib().ar_check_args(R, _ptrs(srcs), _ptrs(dsts), n_dsts, nelem, max_elems,
                               _dtype_code(dst_dtype), _dtype_code(wire_dtype))


def ar_query(key) -> int:
    k = KEYS[key] if isinstance(key, str) else key
    v = ctypes.c_int64(0)
    _check(lib().ar_query(k, ctypes.byref(v)), "ar_query")
    return v.value


def ar_set_option(key, value: int) -> None:
    k = KEYS[key] if isinstance(key, str) else key
    _check(lib().ar_set_option(k, value), "ar_set_option")


def ar_reduce_host(h_srcs, h_dsts, d_srcs=None, d_dsts=None, nelem=None, dst_dtype=None, wire_dtype="bf16",
                   stream=None) -> None:
    """Host partials in, host results out: through the caller's device
    staging buffers, or (``d_srcs``/``d_dsts`` None) with the kernel reading
    and writing the pinned host buffers directly; ordered on ``stream``."""
    nelem, dcode = _infer(d_srcs if d_srcs is not None else h_srcs, nelem, dst_dtype)
    for xs, where in ((h_srcs, "host"), (h_dsts, "host"), (d_srcs, "device"), (d_dsts, "device")):
        _checked(xs, nelem, dcode, where, "ar_reduce_host")
    _check(lib().ar_reduce_host(_ptrs(h_srcs), _ptrs(h_dsts), len(h_dsts), nelem, dcode, _dtype_code(wire_dtype),
                                _ptrs(d_srcs), _ptrs(d_dsts), _stream(stream)), "ar_reduce_host")


def make_layout(ne0, ne1, src_row_bytes=None, dst_row_bytes=None, residual=None, residual_row_bytes=None,
                inactive=()) -> ArLayout:
    """An ar_layout.  With a residual, ``residual_row_bytes`` is its row
    stride in bytes (0: one bias row broadcast to every row; None: packed
    rows, which needs a tensor residual to know the element size);
    ``inactive`` lists rank indices."""
    L = ArLayout()
    L.ne0, L.ne1 = ne0, ne1
    if src_row_bytes is not None:
        L.src_row_bytes = (ctypes.c_int64 * len(src_row_bytes))(*src_row_bytes)
    if dst_row_bytes is not None:
        L.dst_row_bytes = (ctypes.c_int64 * len(dst_row_bytes))(*dst_row_bytes)
    L.residual = _ptr(residual)
    L._residual_obj = residual  # kept for the binding's reach check
    if residual is not None and residual_row_bytes is None:
        residual_row_bytes = ne0 * residual.element_size()
    L.residual_row_bytes = residual_row_bytes or 0
    mask = 0
    for r in inactive:
        mask |= 1 << r
    L.inactive_mask = mask
    return L


def ar_reduce_ex(srcs, dsts, layout: ArLayout, dst_dtype, wire_dtype="bf16", stream=None) -> None:
    """Reduction over an ar_layout (row strides, inactive ranks as None
    sources, residual or bias).  The rows of each CUDA tensor must lie inside
    its storage."""
    es = ESIZE[_dtype_code(dst_dtype)]
    ne0, ne1 = layout.ne0, layout.ne1
    if ne0 * ne1:
        def need(stride):
            return (ne1 - 1) * stride + ne0 * es
        for kind, xs, rows in (("source", srcs, layout.src_row_bytes), ("destination", dsts, layout.dst_row_bytes)):
            for k, x in enumerate(xs):
                reach = _reach(x)
                n = need(rows[k] if rows else ne0 * es)
                if reach is not None and reach < n:
                    raise ValueError(f"ar_reduce_ex: {kind} {k} reaches {reach} bytes, its rows span {n}")
        res = getattr(layout, "_residual_obj", None)
        reach = _reach(res)
        if reach is not None:
            n = ne0 * es if layout.residual_row_bytes == 0 else need(layout.residual_row_bytes)
            if reach < n:
                raise ValueError(f"ar_reduce_ex: the residual reaches {reach} bytes, its rows span {n}")
    _check(lib().ar_reduce_ex(_ptrs(srcs), _ptrs(dsts), len(dsts), ctypes.byref(layout), _dtype_code(dst_dtype),
                              _dtype_code(wire_dtype), _stream(stream)), "ar_reduce_ex")


def ar_check_layout(R, srcs, dsts, layout: ArLayout, max_elems, dst_dtype, wire_dtype) -> int:
    """Host-only validation of an ar_reduce_ex call; returns the status."""
    return lib().ar_check_layout(R, _ptrs(srcs), _ptrs(dsts), len(dsts), ctypes.byref(layout), max_elems,
                                 _dtype_code(dst_dtype), _dtype_code(wire_dtype))


def ar_wire_pack(src, wire, nelem=None, dst_dtype=None, wire_dtype="bf16", stream=None) -> None:
    """wire[i] = T_wire(src[i]): the wire copy a transport would send."""
    if nelem is None:
        nelem = src.numel()
    if dst_dtype is None:
        dst_dtype = src.dtype
    dcode, wcode = _dtype_code(dst_dtype), _dtype_code(wire_dtype)
    _checked([src], nelem, dcode, "device", "ar_wire_pack")
    _checked([wire], nelem, wcode, "device", "ar_wire_pack")
    _check(lib().ar_wire_pack(_ptr(src), _ptr(wire), nelem, _dtype_code(dst_dtype), _dtype_code(wire_dtype),
                              _stream(stream)), "ar_wire_pack")


AR_NOALLOC_SCRATCH_BYTES = 64 << 20


def ar_reduce_host_noalloc(h_srcs, h_dsts, nelem=None, dst_dtype=None, wire_dtype="bf16", stream=None) -> None:
    """Host partials in, host results out, staged through the library's own
    fixed device area: for callers that may not allocate device memory.
    At most AR_NOALLOC_SCRATCH_BYTES of staging per call; calls that overlap
    on the GPU share that area and must not run at the same time."""
    nelem, dcode = _infer(h_srcs, nelem, dst_dtype)
    _checked(h_srcs, nelem, dcode, "host", "ar_reduce_host_noalloc")
    _checked(h_dsts, nelem, dcode, "host", "ar_reduce_host_noalloc")
    _check(lib().ar_reduce_host_noalloc(_ptrs(h_srcs), _ptrs(h_dsts), len(h_dsts), nelem, dcode,
                                        _dtype_code(wire_dtype), _stream(stream)), "ar_reduce_host_noalloc")
