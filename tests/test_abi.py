"""The C ABI without a GPU: the library builds and loads, exports every
function include/ar.h declares, its enums match the binding, and the
host-side argument checks return the documented status codes."""
import ctypes
import os
import re

import pytest
import torch

import tensor_partial_sum_gb300 as tps
from tensor_partial_sum_gb300 import ar as A
from tensor_partial_sum_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "ar.h")
OK, INVALID, UNSUPPORTED, TOO_LARGE, NOT_INIT, OVERLAP, CUDA = range(7)


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(ar_\w+)\s*\(", text, flags=re.M)))


def _enum_values(name_prefix):
    text = open(HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(rf"\b({name_prefix}\w*)\s*=\s*(\d+)", text)}


def test_exports_every_declared_function():
    names = _declared_functions()
    assert {"ar_init", "ar_reduce", "ar_free"} <= set(names)
    lib = ctypes.CDLL(B.LIB)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_enums_match_binding():
    st = _enum_values("AR_OK") | _enum_values("AR_ERR_")
    assert st == {v: k for k, v in A.STATUS_NAMES.items()}
    dt = {k: v for k, v in _enum_values("AR_").items() if k in ("AR_F32", "AR_F16", "AR_BF16")}
    assert dt == {"AR_F32": tps.AR_F32, "AR_F16": tps.AR_F16, "AR_BF16": tps.AR_BF16}
    var = _enum_values("AR_VARIANT_")
    assert {k[len("AR_VARIANT_"):].lower(): v for k, v in var.items()} == A.VARIANTS
    keys = _enum_values("AR_Q_")
    assert {k[len("AR_Q_"):].lower(): v for k, v in keys.items()} == A.KEYS


def test_status_strings():
    for code in range(7):
        s = tps.ar_status_string(code)
        assert s and s != "unknown status"
    assert tps.ar_status_string(99) == "unknown status"


def chk(R=2, srcs=None, dsts=None, n_dsts=None, nelem=64, max_elems=1 << 20, dst="f32", wire="bf16"):
    if srcs is None:
        srcs = [0x10000 * (k + 1) for k in range(R)]
    if dsts is None:
        dsts = [0x100000 * (k + 1) for k in range(2)]
    if n_dsts is None:
        n_dsts = len(dsts)
    return tps.ar_check_args(R, srcs, dsts, n_dsts, nelem, max_elems, dst, wire)


def test_check_args_accepts_good_calls():
    assert chk() == OK
    for d in ("f32", "f16", "bf16"):
        for w in ("f32", "f16", "bf16"):
            assert chk(dst=d, wire=w) == OK
    assert chk(R=16, srcs=[0x10000 * (k + 1) for k in range(16)]) == OK
    assert chk(dsts=[0x1000000 * (k + 1) for k in range(16)]) == OK


def test_check_args_counts():
    assert chk(R=0, srcs=[0x1000]) == INVALID
    assert chk(R=17, srcs=[0x10000 * (k + 1) for k in range(17)]) == INVALID
    assert chk(n_dsts=0) == INVALID
    assert chk(dsts=[0x1000000 * (k + 1) for k in range(17)]) == INVALID


def test_check_args_pointers():
    lib = A.lib()
    assert lib.ar_check_args(2, None, A._ptrs([0x100000]), 1, 64, 100, 0, 2) == INVALID
    assert lib.ar_check_args(2, A._ptrs([0x10000, 0x20000]), None, 1, 64, 100, 0, 2) == INVALID
    assert chk(srcs=[0x10000, 0]) == INVALID
    assert chk(dsts=[0x100000, 0]) == INVALID
    # element alignment: a float pointer must be 4-byte aligned, a half 2-byte
    assert chk(srcs=[0x10002, 0x20000]) == INVALID
    assert chk(srcs=[0x10002, 0x20000], dst="f16") == OK
    assert chk(dsts=[0x100001, 0x200000], dst="bf16") == INVALID
    # nelem == 0 touches nothing, so NULL buffers are fine
    assert chk(srcs=[0, 0], dsts=[0, 0], nelem=0) == OK


def test_check_args_types_and_sizes():
    assert chk(dst=3) == UNSUPPORTED
    assert chk(wire=-1) == UNSUPPORTED
    assert chk(nelem=101, max_elems=100) == TOO_LARGE
    assert chk(nelem=100, max_elems=100) == OK


def test_check_args_overlap():
    n = 64  # 256 bytes of f32
    # a destination exactly equal to a source: in-place, allowed
    assert chk(srcs=[0x10000, 0x20000], dsts=[0x10000], nelem=n) == OK
    # partly overlapping a source
    assert chk(srcs=[0x10000, 0x20000], dsts=[0x10000 + 128], nelem=n) == OVERLAP
    assert chk(srcs=[0x10000, 0x20000], dsts=[0x20000 - 128], nelem=n) == OVERLAP
    # adjacent, not overlapping
    assert chk(srcs=[0x10000, 0x20000], dsts=[0x10000 + 256], nelem=n) == OK
    # two destinations that meet, or are the same buffer
    assert chk(dsts=[0x100000, 0x100000 + 128], nelem=n) == OVERLAP
    assert chk(dsts=[0x100000, 0x100000], nelem=n) == OVERLAP
    # sources may overlap each other (they are only read)
    assert chk(srcs=[0x10000, 0x10000 + 128], nelem=n) == OK


def test_check_args_overlap_on_host_arrays():
    """The same rule guards the host buffers of ar_reduce_host and
    ar_reduce_host_noalloc (they run it on the host pointers): views of one
    numpy buffer that partly overlap are refused, an exact alias is not."""
    import numpy as np
    n = 1000
    back = np.zeros(3 * n, dtype=np.float32)
    srcs = [back[:n], back[2 * n:]]
    assert chk(srcs=srcs, dsts=[back[n // 2:n // 2 + n]], nelem=n) == OVERLAP
    assert chk(srcs=srcs, dsts=[back[n:2 * n]], nelem=n) == OK
    assert chk(srcs=srcs, dsts=[srcs[1]], nelem=n) == OK
    other = np.zeros(2 * n, dtype=np.float32)
    assert chk(srcs=srcs, dsts=[other[:n], other[n - 1:2 * n - 1]], nelem=n) == OVERLAP


def test_calls_before_init():
    tps.ar_free()
    tps.ar_free()  # a second free is harmless
    lib = A.lib()
    v = ctypes.c_int64()
    assert lib.ar_query(0, ctypes.byref(v)) == NOT_INIT
    assert lib.ar_set_option(4, 1) == NOT_INIT
    s, d = A._ptrs([0x10000, 0x20000]), A._ptrs([0x100000])
    assert lib.ar_reduce(s, d, 1, 64, 0, 2, None) == NOT_INIT
    assert lib.ar_reduce_variant(s, d, 1, 64, 0, 2, 2, 0, None) == NOT_INIT
    assert lib.ar_reduce_host(s, d, 1, 64, 0, 2, s, d, None) == NOT_INIT


def test_init_argument_errors():
    lib = A.lib()
    assert lib.ar_init(0, 100) == INVALID
    assert lib.ar_init(17, 100) == INVALID
    assert lib.ar_init(2, 0) == INVALID


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_init_without_a_device_reports_cuda():
    assert A.lib().ar_init(2, 100) == CUDA


def test_binding_raises_on_error():
    tps.ar_free()
    with pytest.raises(tps.ARError) as e:
        tps.ar_query("ranks")
    assert e.value.status == NOT_INIT


def lay(**kw):
    return tps.make_layout(**kw)


def chk_l(R=2, srcs=None, dsts=None, max_elems=1 << 20, dst="f32", wire="bf16", **kw):
    if srcs is None:
        srcs = [0x1000000 * (k + 1) for k in range(R)]
    if dsts is None:
        dsts = [0x40000000]
    kw.setdefault("ne0", 64)
    kw.setdefault("ne1", 4)
    return tps.ar_check_layout(R, srcs, dsts, lay(**kw), max_elems, dst, wire)


def test_check_layout_basics():
    assert chk_l() == OK
    assert chk_l(ne0=0) == OK and chk_l(ne1=0) == OK  # empty: nothing touched
    assert chk_l(ne0=1024, ne1=1025, max_elems=1 << 20) == TOO_LARGE
    assert chk_l(dst=5) == UNSUPPORTED
    assert chk_l(srcs=[0x1000000, 0]) == INVALID
    assert chk_l(srcs=[0x1000002, 0x2000000]) == INVALID  # misaligned f32


def test_check_layout_strides():
    assert chk_l(src_row_bytes=[256, 512]) == OK
    assert chk_l(src_row_bytes=[255, 256]) == INVALID    # shorter than a row (64 x 4 bytes)
    assert chk_l(src_row_bytes=[258, 256]) == INVALID    # not a multiple of the element size
    assert chk_l(dst_row_bytes=[300]) == OK
    assert chk_l(dst_row_bytes=[100]) == INVALID
    assert chk_l(ne1=1, src_row_bytes=[0, 0]) == OK      # one row: the stride is never used


def test_check_layout_inactive_ranks():
    assert chk_l(srcs=[0x1000000, 0], inactive=(1,)) == OK     # NULL allowed for an inactive rank
    assert chk_l(srcs=[0, 0], inactive=(0, 1)) == OK
    assert chk_l(inactive=(2,)) == INVALID                    # bit beyond R


def test_check_layout_residual_and_overlap():
    n = 64 * 4 * 4  # bytes of one 64 x 4 f32 tensor
    assert chk_l(residual=0x3000000, residual_row_bytes=256) == OK
    assert chk_l(residual=0x3000000, residual_row_bytes=0) == OK      # bias row
    assert chk_l(residual=0x3000000, residual_row_bytes=200) == INVALID
    # in place into the residual: same pointer, same stride
    assert chk_l(residual=0x40000000, residual_row_bytes=256) == OK
    assert chk_l(residual=0x40000000, residual_row_bytes=512, dst_row_bytes=[256]) == OVERLAP
    # destination into a broadcast bias row: overlap
    assert chk_l(residual=0x40000000, residual_row_bytes=0) == OVERLAP
    # in place into a source, and a partial overlap
    assert chk_l(dsts=[0x1000000]) == OK
    assert chk_l(dsts=[0x1000000 + 128]) == OVERLAP
    assert chk_l(dsts=[0x1000000 + n]) == OK
    # two destinations overlapping
    assert chk_l(dsts=[0x40000000, 0x40000000 + 64]) == OVERLAP
    # an inactive rank's pointer is never read, so it cannot overlap
    assert chk_l(srcs=[0x1000000, 0x40000000 + 8], inactive=(1,)) == OK


def test_every_environment_knob_is_documented():
    """Each environment variable the library reads is described in the header."""
    src = open(os.path.join(os.path.dirname(HEADER), "..", "tensor_partial_sum_gb300", "csrc", "ar.cu")).read()
    names = set(re.findall(r'(?:getenv|env_int)\("([A-Z_]+)"', src))
    assert {"AR_VARIANT", "AR_PDL"} <= names
    header = open(HEADER).read()
    missing = [n for n in sorted(names) if n not in header]
    assert not missing, missing
