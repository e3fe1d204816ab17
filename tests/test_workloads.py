"""The seeded input generators draw what the design states: same seed, same
bytes; ranks independent; and the stated value distributions (checked on
samples with tolerances several standard errors wide)."""
import numpy as np
import pytest

from tensor_partial_sum_gb300 import workloads as W
from tests.libcasts import lib_widen

N = 1 << 20


def test_deterministic_and_ranks_differ():
    for name in W.WORKLOADS:
        a = W.generate(name, nelem=4096)
        b = W.generate(name, nelem=4096)
        assert all(np.array_equal(x, y) for x, y in zip(a, b)), name
        if W.WORKLOADS[name].R > 1:
            assert not np.array_equal(a[0], a[1]), name


def test_shapes_and_bytes():
    w = W.WORKLOADS["prefill"]
    assert (w.R, w.n_dsts, w.nelem, w.dst, w.wire) == (2, 2, 2048 * 4096, "f32", "bf16")
    assert w.bytes_per_call == 4 * 2048 * 4096 * 4
    d = W.WORKLOADS["decode"]
    assert (d.R, d.n_dsts, d.nelem, d.calls, d.wire) == (4, 4, 4099, 10000, "f16")
    assert W.WORKLOADS["f16_edges"].bytes_per_call == 9 * 8192 * 8192 * 4
    assert W.WORKLOADS["prefill_inactive"].bytes_per_call == 3 * 2048 * 4096 * 4
    assert W.WORKLOADS["prefill_residual"].bytes_per_call == 5 * 2048 * 4096 * 4
    assert W.WORKLOADS["prefill_pack"].bytes_per_call == 2048 * 4096 * (4 + 2)


def test_decode_calls_use_their_own_seeds():
    a = W.generate("decode", call=0)
    b = W.generate("decode", call=1)
    assert a[0].size == 4099 and not np.array_equal(a[0], b[0])
    x = np.concatenate([W.generate("decode", call=k)[0] for k in range(64)])
    assert abs(x.std() - 0.5) < 0.02 and abs(x.mean()) < 0.02


def test_normal_and_prefill_outliers():
    (x, _) = W.generate("tp_small", nelem=N)
    assert abs(x.std() - 1.0) < 0.01
    p = W.generate("prefill", nelem=N)[0]
    frac = np.mean(np.abs(p) > 8.0)  # N(0,1) beyond 8 sigma: never; x50 outliers: mostly
    assert 0.0007 < frac < 0.0013


def test_student_t3_scaled():
    b = W.generate("bf16_t3", nelem=N)[0]
    v = lib_widen("bf16", b).astype(np.float64)
    # median |t_3| = 0.7649; times 0.2
    assert abs(np.median(np.abs(v)) - 0.2 * 0.7649) < 0.005
    # heavy tails: P(|t_3| > 5) = 0.01540, so P(|v| > 1) = 0.0154
    assert abs(np.mean(np.abs(v) > 1.0) - 0.0154) < 0.002


def test_f16_edge_mixture_and_planted_values():
    x = W.generate("f16_edges", nelem=N)
    a = np.abs(x[0].astype(np.float64))
    big = np.mean((a >= 5.4e4) & (a <= 6.6e4))
    tiny = np.mean((a >= 1e-7) & (a <= 6e-5))
    assert abs(big - 0.01) < 0.001 and 0.0095 < tiny < 0.0115  # N(0,1) adds a few tiny ones
    assert np.isin(np.float32(65520.0), x[0][:8]) and np.isin(np.float32(2.0 ** -24), x[0][:8])
    assert np.signbit(x[1][:8]).any()  # -0 and negative edges are planted too
    assert not np.array_equal(x[0][:8], x[1][:8])  # rolled per rank


@pytest.mark.parametrize("name", ["prefill_residual", "prefill_bias"])
def test_residual_drawn_after_the_ranks(name):
    w = W.WORKLOADS[name]
    arrs = W.generate(w, nelem=8192)
    assert len(arrs) == w.R + 1
    assert arrs[-1].size == (w.ne0 if w.residual == "row" else 8192)
