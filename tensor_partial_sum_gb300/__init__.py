"""GB300-native partial-sum reduction (the reduction step of a
tensor-parallel AllReduce) behind a small C ABI.

The compute path is ``libtps_ar.so`` (hand-written CUDA for sm_103a);
``tensor_partial_sum_gb300.ar`` is a ctypes binding with the same names as
the C entry points.  The first call fails loudly (RuntimeError) when the
library is not built; there is no other implementation to fall back to.
"""
from .ar import (  # noqa: F401
    AR_BF16, AR_F16, AR_F32, ARError, DTYPE_CODES, ar_check_args, ar_free, ar_init,
    ar_query, ar_reduce, ar_reduce_host, ar_reduce_variant, ar_set_option,
    ar_status_string, library_path, ArLayout, make_layout, ar_reduce_ex, ar_check_layout, ar_wire_pack,
    ar_reduce_host_noalloc, AR_NOALLOC_SCRATCH_BYTES, PreparedReduce,
)
