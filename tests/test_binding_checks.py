"""The Python binding refuses buffers that a kernel would read or write past
their end, or in the wrong memory, before any address reaches the library
(CPU only: every case raises before the C call)."""
import numpy as np
import pytest
import torch

import tensor_partial_sum_gb300 as tps


def test_device_entry_points_refuse_host_tensors():
    a = torch.zeros(64)
    with pytest.raises(TypeError, match="cpu tensor"):
        tps.ar_reduce([a, a], [a.clone()], wire_dtype="bf16")
    with pytest.raises(TypeError, match="numpy array"):
        tps.ar_reduce_variant([np.zeros(64, np.float32)] * 2, [np.zeros(64, np.float32)], "latency",
                              dst_dtype="f32")
    with pytest.raises(TypeError, match="cpu tensor"):
        tps.ar_wire_pack(a, torch.zeros(64, dtype=torch.bfloat16))


def test_non_contiguous_and_short_buffers_are_refused():
    a = torch.zeros(8, 8).t()  # a transposed view: not contiguous
    with pytest.raises(ValueError, match="not contiguous"):
        tps.ar_reduce_host([a, a], [torch.zeros(64)], dst_dtype="f32")
    short = np.zeros(10, np.float32)
    full = np.zeros(64, np.float32)
    with pytest.raises(ValueError, match="holds 40 bytes, the call needs 256"):
        tps.ar_reduce_host_noalloc([full, full], [short], nelem=64, dst_dtype="f32")
    with pytest.raises(ValueError, match="not contiguous"):
        tps.ar_reduce_host_noalloc([full[::2], full[::2]], [full[:32].copy()], dst_dtype="f32")


def test_device_staging_must_be_device_memory():
    h = [np.zeros(64, np.float32) for _ in range(2)]
    with pytest.raises(TypeError, match="device buffer is needed"):
        tps.ar_reduce_host(h, [np.zeros(64, np.float32)], d_srcs=h, d_dsts=[np.zeros(64, np.float32)],
                           dst_dtype="f32")


def test_the_wire_buffer_is_sized_in_wire_elements():
    """A bf16 wire copy of 64 f32 elements needs 128 bytes, not 256."""
    src = np.zeros(64, np.float32)
    wire_ok = np.zeros(64, np.uint16)
    from tensor_partial_sum_gb300 import ar
    ar._checked([wire_ok], 64, ar.AR_BF16, "host", "t")
    with pytest.raises(ValueError):
        ar._checked([np.zeros(63, np.uint16)], 64, ar.AR_BF16, "host", "t")
    ar._checked([src], 64, ar.AR_F32, "host", "t")
    ar._checked([12345, None], 64, ar.AR_F32, "device", "t")  # raw addresses pass unchecked


def test_reach_needs_a_cuda_tensor():
    """Raw addresses are not checked; host tensors are refused (the reach of
    CUDA views is tested on the GPU)."""
    from tensor_partial_sum_gb300 import ar
    assert ar._reach(None) is None and ar._reach(1234) is None
    with pytest.raises(TypeError):
        ar._reach(torch.zeros(8))


def test_ex_refuses_rows_past_the_storage_on_cpu_tensors():
    a = torch.zeros(64)
    lay = tps.make_layout(8, 8)
    with pytest.raises(TypeError):
        tps.ar_reduce_ex([a, a], [a.clone()], lay, "f32")


def test_prepared_call_checks_its_buffers_once():
    a = torch.zeros(64)
    with pytest.raises(TypeError, match="cpu tensor"):
        tps.PreparedReduce([a, a], [a.clone()])


def test_pointer_arrays_are_packed_addresses():
    """Pointer arrays reach the library as native 64-bit addresses, padded
    with NULLs to 16 entries (so a short list reads as a NULL source, which
    the library refuses, instead of memory past the list)."""
    import struct
    from tensor_partial_sum_gb300 import ar
    packed = ar._ptrs([0x1000, None, 0xFFFFFFFFFFFFFFF0])
    assert len(packed) == 16 * 8
    vals = struct.unpack("=16Q", packed)
    assert vals[:3] == (0x1000, 0, 0xFFFFFFFFFFFFFFF0) and vals[3:] == (0,) * 13
    assert ar._ptrs(None) is None
    assert len(ar._ptrs(list(range(1, 18)))) == 17 * 8
    a = np.zeros(4, np.float32)
    assert struct.unpack("=16Q", ar._ptrs([a]))[0] == a.ctypes.data
