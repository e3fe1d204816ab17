"""Helpers shared by the GPU tests: move storage arrays to and from the
device and run one reduction through the C ABI."""
import numpy as np
import torch

import tensor_partial_sum_gb300 as tps

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ESIZE = {"f32": 4, "f16": 2, "bf16": 2}


def to_device(a: np.ndarray, name: str) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if name == "f32":
        return torch.from_numpy(a.view(np.float32)).cuda()
    t = torch.from_numpy(a.view(np.int16)).cuda()
    return t.view(TORCH_DTYPE[name])


def to_host(t: torch.Tensor, name: str) -> np.ndarray:
    t = t.detach().contiguous()
    if name == "f32":
        return t.cpu().numpy().view(np.float32).ravel()
    return t.view(torch.int16).cpu().numpy().view(np.uint16).ravel()


class Ctx:
    """Keeps one library context alive and re-initialises it when R or the
    size limit grows."""

    def __init__(self):
        self.R = None
        self.max_elems = 0

    def ensure(self, R, nelem):
        if self.R != R or nelem > self.max_elems:
            self.max_elems = max(nelem, 1 << 16)
            tps.ar_init(R, self.max_elems)
            self.R = R


def empty_like_poisoned(n, name, pad=0, poison=0x7F):
    """A device buffer of n elements with ``pad`` poisoned bytes on each side
    (returns the backing byte tensor and the element view)."""
    es = ESIZE[name]
    back = torch.full((n * es + 2 * pad,), poison, dtype=torch.uint8, device="cuda")
    view = back[pad:pad + n * es].view(TORCH_DTYPE[name])
    return back, view


def run(ctx, srcs_np, n_dsts, dst, wire, variant="auto", grid=0, src_offsets=None, dst_offsets=None,
        pad=0, in_place=None):
    """Run one reduction on the GPU.  Offsets (in elements) shift buffers off
    16-byte alignment.  ``in_place=k`` makes destination 0 be source k.
    Returns (list of destination arrays, list of poisoned backing buffers)."""
    R = len(srcs_np)
    n = srcs_np[0].size
    ctx.ensure(R, n)
    es = ESIZE[dst]
    src_offsets = src_offsets or [0] * R
    dst_offsets = dst_offsets or [0] * n_dsts
    src_t, keep = [], []
    for a, off in zip(srcs_np, src_offsets):
        back = torch.zeros((n + off) * es + 16, dtype=torch.uint8, device="cuda")
        view = back[off * es:(off + n) * es].view(TORCH_DTYPE[dst])
        view.copy_(to_device(a, dst))
        src_t.append(view)
        keep.append(back)
    dst_t, backs = [], []
    for off in dst_offsets:
        back, view = empty_like_poisoned(n + off, dst, pad)
        view = view[off:]
        dst_t.append(view)
        backs.append((back, pad, (n + off) * es, off * es))
    if in_place is not None:
        dst_t[0] = src_t[in_place]
    stream = torch.cuda.current_stream()
    tps.ar_reduce_variant([t.data_ptr() for t in src_t], [t.data_ptr() for t in dst_t], variant, grid,
                          nelem=n, dst_dtype=tps.DTYPE_CODES[dst], wire_dtype=wire, stream=stream)
    torch.cuda.synchronize()
    outs = [to_host(t, dst) for t in dst_t]
    return outs, backs


def check_guards(backs, poison=0x7F):
    """The poisoned margins around each destination are untouched."""
    for back, pad, nbytes, lead in backs:
        if pad == 0 and lead == 0:
            continue
        b = back.cpu().numpy()
        assert (b[:pad + lead] == poison).all(), "bytes before a destination were written"
        assert (b[pad + nbytes:] == poison).all(), "bytes after a destination were written"
