"""Randomised checks of the C ABI's host-side validation (no GPU): for many
generated calls, ar_check_args and ar_check_layout return the status that
the rules of include/ar.h give, taken in the order the header lists them.
The model below restates those rules; the library is not consulted to
build it."""
import pytest

from tensor_partial_sum_gb300 import ar as A

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

OK, INVALID, UNSUPPORTED, TOO_LARGE, OVERLAP = 0, 1, 2, 3, 5
ESIZE = {0: 4, 1: 2, 2: 2}


def overlaps(a, b, n):
    return a < b + n and b < a + n


def model_check_args(R, srcs, dsts, n_dsts, nelem, max_elems, dst, wire):
    """Status of one ar_reduce call by the header's rules, in its order."""
    if not 1 <= R <= 16 or not 1 <= n_dsts <= 16:
        return INVALID
    if dst not in ESIZE or wire not in ESIZE:
        return UNSUPPORTED
    if nelem > max_elems:
        return TOO_LARGE
    if nelem == 0:
        return OK
    es = ESIZE[dst]
    for p in srcs[:R]:
        if not p or p % es:
            return INVALID
    for p in dsts[:n_dsts]:
        if not p or p % es:
            return INVALID
    nb = nelem * es
    for d in range(n_dsts):
        a = dsts[d]
        for r in range(R):
            if a != srcs[r] and overlaps(a, srcs[r], nb):
                return OVERLAP
        for e in range(d):
            if overlaps(a, dsts[e], nb):
                return OVERLAP
    return OK


# pointers drawn from a small window so that overlaps, exact aliases and
# misaligned addresses all come up often
ptr = st.one_of(st.just(0), st.integers(min_value=0x10000, max_value=0x10000 + 512))


@settings(max_examples=3000, deadline=None)
@given(R=st.integers(0, 17), n_dsts=st.integers(0, 17), srcs=st.lists(ptr, min_size=17, max_size=17),
       dsts=st.lists(ptr, min_size=17, max_size=17), nelem=st.integers(0, 80),
       max_elems=st.integers(0, 100), dst=st.integers(0, 3), wire=st.integers(0, 3))
def test_check_args_follows_the_rules(R, n_dsts, srcs, dsts, nelem, max_elems, dst, wire):
    got = A.lib().ar_check_args(R, A._ptrs(srcs[:max(R, 1)]), A._ptrs(dsts[:max(n_dsts, 1)]), n_dsts, nelem,
                                max_elems, dst, wire)
    # _ptrs pads to 16 entries with NULL; beyond that the model reads the same lists
    want = model_check_args(R, srcs[:max(R, 1)] + [0] * 17, dsts[:max(n_dsts, 1)] + [0] * 17, n_dsts, nelem,
                            max_elems, dst, wire)
    assert got == want


@settings(max_examples=1500, deadline=None)
@given(R=st.integers(1, 4), srcs=st.lists(st.integers(0x10000, 0x10000 + 256).map(lambda x: x & ~3), min_size=4,
                                          max_size=4),
       dsts=st.lists(st.integers(0x10000, 0x10000 + 256).map(lambda x: x & ~3), min_size=2, max_size=2),
       n_dsts=st.integers(1, 2), ne0=st.integers(0, 8), ne1=st.integers(0, 4), stride_extra=st.integers(0, 4),
       inactive=st.integers(0, 15))
def test_check_layout_overlap_rules(R, srcs, dsts, n_dsts, ne0, ne1, stride_extra, inactive):
    """Row-strided f32 layouts: a destination may be exactly an active
    source with the same stride; any other overlap of row spans is
    refused; inactive ranks are never looked at."""
    inactive &= (1 << R) - 1
    stride = (ne0 + stride_extra) * 4
    lay = A.ArLayout()
    lay.ne0, lay.ne1 = ne0, ne1
    import ctypes
    lay.src_row_bytes = (ctypes.c_int64 * R)(*([stride] * R))
    lay.dst_row_bytes = (ctypes.c_int64 * n_dsts)(*([stride] * n_dsts))
    lay.inactive_mask = inactive
    s = [0 if (inactive >> r) & 1 else srcs[r] for r in range(R)]
    got = A.lib().ar_check_layout(R, A._ptrs(s), A._ptrs(dsts[:n_dsts]), n_dsts, ctypes.byref(lay), 1 << 20, 0, 2)
    if ne0 * ne1 == 0:
        assert got == OK
        return
    span = (ne1 - 1) * stride + ne0 * 4 if ne1 > 1 else ne0 * 4
    want = OK
    for d in range(n_dsts):
        for r in range(R):
            if (inactive >> r) & 1:
                continue
            if overlaps(dsts[d], s[r], span) and dsts[d] != s[r]:
                want = OVERLAP
        for e in range(d):
            if overlaps(dsts[d], dsts[e], span):
                want = OVERLAP
    assert got == want
