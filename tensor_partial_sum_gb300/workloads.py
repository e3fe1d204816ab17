"""Seeded synthetic workloads: R partial tensors shaped like the activations
a tensor-parallel AllReduce sums during decode and prefill.

This module only draws input data.  It holds none of the reduction's
arithmetic and is the one piece shared by the library's tests, the oracle
checks and the benchmark.  Random draws use numpy's PCG64 generator; rank r
draws from the r-th child stream that ``SeedSequence(seed).spawn(R)`` gives
(so ranks can be drawn in parallel and still be reproducible).  Arrays are
returned in storage form: ``float32`` for f32, ``uint16`` bit patterns for
f16/bf16.

The five workloads (sizes as the reduction sees them):

========== === ====== ============== ================== ====== ==========
name         R n_dsts T_dst / T_wire shape              seed   values
========== === ====== ============== ================== ====== ==========
tp_small     2      2 f32 / bf16     [32, 4096]         0      N(0, 1)
decode       4      4 f32 / f16      [1, 4099] x 10000  1000+k N(0, 0.5)
prefill      2      2 f32 / bf16     [2048, 4096]       3      N(0, 1), 0.1% x50
bf16_t3      4      4 bf16 / bf16    [4096, 8192]       4      bf16(0.2 t(3))
f16_edges    8      1 f32 / f16      [8192, 8192]       5      mixture, below
========== === ====== ============== ================== ====== ==========

f16_edges draws each element from: 98% N(0, 1); 1% +-U(5.4e4, 6.6e4), which
straddles binary16's overflow threshold 65520, so some wire values become
+-inf and some sums NaN; 1% +-logU(1e-7, 6e-5), binary16's subnormal range.
It also plants exact edge values (+-0, 65504, 65520, 2^-24, 2^-25) at the
first and last eight positions of every rank.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
import os

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    n_dsts: int
    dst: str
    wire: str
    shape: tuple
    seed: int
    values: str
    calls: int = 1
    # extended layouts (ar_reduce_ex) and the wire pack
    op: str = "reduce"            # "reduce", "reduce_ex" or "pack"
    residual: str = ""            # "", "full" (a residual tensor) or "row" (one bias row)
    row_pad: int = 0              # extra elements between rows (row stride = shape[-1] + row_pad)
    inactive: tuple = ()          # ranks that contribute +0

    @property
    def ne0(self) -> int:
        return self.shape[-1]

    @property
    def ne1(self) -> int:
        return self.nelem // self.shape[-1]

    @property
    def nelem(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dst == "f32" else 2

    @property
    def bytes_per_call(self) -> int:
        """Algorithmic bytes: every active source (and the residual) read
        once, every destination written once; row padding is not touched."""
        es = self.elem_bytes
        if self.op == "pack":
            return self.nelem * es + self.nelem * (4 if self.wire == "f32" else 2)
        n = (self.R - len(self.inactive) + self.n_dsts) * self.nelem * es
        if self.residual == "full":
            n += self.nelem * es
        elif self.residual == "row":
            n += self.ne0 * es
        return n

    def describe(self) -> str:
        shape = "x".join(str(s) for s in self.shape)
        calls = f" x{self.calls} calls" if self.calls > 1 else ""
        if self.op == "pack":
            return f"wire pack {self.dst}[{shape}] -> {self.wire} values={self.values}"
        extra = ""
        if self.residual:
            extra += f" residual={self.residual}"
        if self.row_pad:
            extra += f" row_stride={self.ne0 + self.row_pad}"
        if self.inactive:
            extra += f" inactive={list(self.inactive)}"
        return (f"R={self.R} {self.dst}[{shape}]{calls} wire={self.wire} n_dsts={self.n_dsts} "
                f"values={self.values}{extra}")


WORKLOADS = {
    w.name: w for w in [
        Workload("tp_small", 2, 2, "f32", "bf16", (32, 4096), 0, "normal(0,1)"),
        Workload("decode", 4, 4, "f32", "f16", (1, 4099), 1000, "normal(0,0.5)", calls=10000),
        Workload("prefill", 2, 2, "f32", "bf16", (2048, 4096), 3, "normal(0,1)+0.1%x50"),
        Workload("bf16_t3", 4, 4, "bf16", "bf16", (4096, 8192), 4, "bf16(0.2*t3)"),
        Workload("f16_edges", 8, 1, "f32", "f16", (8192, 8192), 5, "f16-edge mixture"),
        # the prefill shape through the extended entry points
        Workload("prefill_residual", 2, 2, "f32", "bf16", (2048, 4096), 3, "normal(0,1)+0.1%x50",
                 op="reduce_ex", residual="full"),
        Workload("prefill_bias", 2, 2, "f32", "bf16", (2048, 4096), 3, "normal(0,1)+0.1%x50",
                 op="reduce_ex", residual="row"),
        Workload("prefill_strided", 2, 2, "f32", "bf16", (2048, 4096), 3, "normal(0,1)+0.1%x50",
                 op="reduce_ex", row_pad=64),
        Workload("prefill_inactive", 2, 2, "f32", "bf16", (2048, 4096), 3, "normal(0,1)+0.1%x50",
                 op="reduce_ex", inactive=(1,)),
        Workload("prefill_pack", 1, 1, "f32", "bf16", (2048, 4096), 3, "normal(0,1)+0.1%x50", op="pack"),
    ]
}

PLANTED = np.array([0.0, -0.0, 65504.0, 65520.0, 2.0 ** -24, 2.0 ** -25, -65520.0, -(2.0 ** -24)],
                   dtype=np.float32)


def _normal(rng, n, sigma):
    x = rng.standard_normal(n, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return x


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 storage via torch's conversion (input synthesis
    only; the reduction never calls this)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rank(w: Workload, rng, n: int, r: int) -> np.ndarray:
    if w.values == "normal(0,1)":
        return _normal(rng, n, 1.0)
    if w.values == "normal(0,0.5)":
        return _normal(rng, n, 0.5)
    if w.values == "normal(0,1)+0.1%x50":
        x = _normal(rng, n, 1.0)
        hit = rng.random(n, dtype=np.float32) < np.float32(0.001)
        x[hit] *= np.float32(50.0)
        return x
    if w.values == "bf16(0.2*t3)":
        # Student t with 3 degrees of freedom: Z0 / sqrt((Z1^2 + Z2^2 + Z3^2) / 3)
        z0 = rng.standard_normal(n, dtype=np.float32)
        v = np.zeros(n, dtype=np.float32)
        for _ in range(3):
            z = rng.standard_normal(n, dtype=np.float32)
            v += z * z
        v *= np.float32(1.0 / 3.0)
        np.sqrt(v, out=v)
        z0 /= v
        z0 *= np.float32(0.2)
        return _to_bf16_bits(z0)
    if w.values == "f16-edge mixture":
        x = _normal(rng, n, 1.0)
        u = rng.random(n, dtype=np.float32)
        big = np.nonzero((u >= np.float32(0.98)) & (u < np.float32(0.99)))[0]
        tiny = np.nonzero(u >= np.float32(0.99))[0]
        sb = np.where(rng.random(big.size) < 0.5, -1.0, 1.0)
        x[big] = (sb * rng.uniform(5.4e4, 6.6e4, big.size)).astype(np.float32)
        st = np.where(rng.random(tiny.size) < 0.5, -1.0, 1.0)
        x[tiny] = (st * np.exp(rng.uniform(np.log(1e-7), np.log(6e-5), tiny.size))).astype(np.float32)
        k = PLANTED.size
        if n >= 2 * k:
            rolled = np.roll(PLANTED, r)
            x[:k] = rolled
            x[n - k:] = rolled[::-1]
        return x
    raise KeyError(w.values)


def generate(w: Workload | str, call: int = 0, nelem: int | None = None) -> list:
    """The R source arrays of one call (``call`` selects the per-call seed of
    multi-call workloads).  ``nelem`` draws a shorter prefix-shaped sample
    with the same recipe (used for small test cases).  Workloads with a
    residual get it as one more array after the R sources (a full tensor,
    or one row for a bias)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    n = w.nelem if nelem is None else nelem
    seed = w.seed + call if w.calls > 1 else w.seed
    streams = np.random.SeedSequence(seed).spawn(w.R)

    def one(r):
        return _rank(w, np.random.Generator(np.random.PCG64(streams[r])), n, r)

    if n * w.R < (1 << 22):
        out = [one(r) for r in range(w.R)]
    else:
        with ThreadPoolExecutor(max_workers=min(w.R, os.cpu_count() or 1)) as ex:
            out = list(ex.map(one, range(w.R)))
    if w.residual:
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(w.R + 1)[w.R]))
        out.append(_rank(w, rng, w.ne0 if w.residual == "row" else n, w.R))
    return out
