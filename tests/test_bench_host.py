"""bench.py's host-side helpers without a GPU: the clock summary, the
throttle rule, and reading traffic from the committed ncu summary."""
import datetime as dt
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def rows(spec):
    t0 = dt.datetime(2026, 1, 1, 12, 0, 0)
    return [{"t": t0 + dt.timedelta(seconds=s), "sm": mhz, "max": 2070.0, "reasons": rs} for s, mhz, rs in spec]


def test_summary_uses_samples_inside_the_timed_region():
    r = rows([(0, 1000.0, []), (1, 2070.0, []), (2, 2060.0, ["sw_power_cap"]), (3, 2070.0, []), (9, 500.0, [])])
    t0 = dt.datetime(2026, 1, 1, 12, 0, 1)
    t1 = dt.datetime(2026, 1, 1, 12, 0, 3)
    c = bench.ClockSampler.summarize(r, t0, t1)
    assert c["samples"] == 3 and c["window"] == "timed region"
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    assert not bench.throttled(c)


def test_short_region_falls_back_to_all_samples_and_throttle_rule():
    r = rows([(0, 1500.0, ["hw_thermal_slowdown"]), (1, 1500.0, [])])
    t = dt.datetime(2026, 1, 1, 12, 0, 0, 500000)
    c = bench.ClockSampler.summarize(r, t, t)
    assert c["window"].startswith("sustained") and c["samples"] == 2
    assert bench.throttled(c)
    assert bench.ClockSampler.summarize([], t, t)["samples"] == 0


def test_traffic_field_follows_the_kernel_sources():
    v = bench.traffic_per_launch("prefill")
    text = open(bench.TRAFFIC_SUMMARY).read()
    recorded = [l for l in text.splitlines() if l.startswith("- source_digest:")][0]
    if bench.sources_digest() in recorded:
        assert isinstance(v, int) and v > 100_000_000
    else:
        assert v is None  # the kernel changed since the counters were taken
    assert bench.traffic_per_launch("decode") is None


def test_aggregate():
    assert bench.aggregate_gbs(134217728, 100, 2, 0.001) == 2 * 134217728 * 100 / 0.001 / 1e9


def test_digest_ignores_comments_and_whitespace():
    a = "int f(int x) { // add one\n  return x + 1; /* done */ }\n"
    b = "int f(int x) {\n\n    return x + 1;   }"
    assert bench.code_tokens(a) == bench.code_tokens(b)
    assert bench.code_tokens(a) != bench.code_tokens(a.replace("x + 1", "x + 2"))


def test_oracle_row_ranges_tile_the_step():
    """The threaded CPU baseline splits a step into contiguous row ranges:
    their results, laid end to end, are the whole step's bytes, for every
    kind of step the workloads have."""
    import numpy as np
    from tensor_partial_sum_gb300 import workloads as W
    for name in ["tp_small", "prefill_bias", "prefill_inactive", "prefill_pack"]:
        w = W.WORKLOADS[name]
        srcs = W.generate(w)
        whole = bench.oracle_step(w, srcs, 0, 40)
        parts = [bench.oracle_step(w, srcs, a, b) for a, b in [(0, 13), (13, 14), (14, 40)]]
        if w.op == "pack":
            assert np.array_equal(whole.view(np.uint8), np.concatenate(parts).view(np.uint8)), name
        else:
            for d in range(w.n_dsts):
                cat = np.concatenate([p[d] for p in parts])
                assert np.array_equal(whole[d].view(np.uint8), cat.view(np.uint8)), (name, d)


def test_oracle_rate_reports_its_threads():
    from tensor_partial_sum_gb300 import workloads as W
    w = W.WORKLOADS["tp_small"]
    v, el, text = bench.oracle_rate(W.generate(w), w, 0.2, steps=2, threads=2)
    assert v > 0 and el > 0 and "on 2 thread(s)" in text
