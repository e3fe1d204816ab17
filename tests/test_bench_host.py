"""bench.py's host-side helpers without a GPU: the clock summary, the
throttle rule, reading traffic from the committed ncu counters, the
roofline record and the step counts of the workloads measured beside the
headline."""
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


def test_traffic_field_follows_the_kernel_sources(tmp_path):
    import json
    recorded = json.load(open(bench.TRAFFIC_FILE))["workloads"]
    assert {"tp_small", "prefill", "bf16_t3", "f16_edges"} <= set(recorded)
    for name, e in recorded.items():
        v = bench.traffic_per_launch(name)
        # no launch moves more than its algorithmic bytes (nothing read twice); writes may
        # trail them while destinations are still dirty in L2
        assert e["dram_bytes_per_launch"] <= 1.01 * e["algorithmic_bytes_per_launch"], name
        if e["source_digest"] == bench.sources_digest():
            assert v == e["dram_bytes_per_launch"]
        else:
            assert v is None  # the kernel changed since the counters were taken
    assert bench.traffic_per_launch("decode") is None
    # a stale digest, a missing file and a malformed file all read as "no figure"
    p = tmp_path / "t.json"
    p.write_text(json.dumps({"workloads": {"prefill": {"source_digest": "0", "dram_bytes_per_launch": 5}}}))
    assert bench.traffic_per_launch("prefill", str(p)) is None
    p.write_text(json.dumps({"workloads": {"prefill": {"source_digest": bench.sources_digest(),
                                                       "dram_bytes_per_launch": 5}}}))
    assert bench.traffic_per_launch("prefill", str(p)) == 5
    assert bench.traffic_per_launch("prefill", str(tmp_path / "none.json")) is None
    p.write_text("not json")
    assert bench.traffic_per_launch("prefill", str(p)) is None


def test_config_steps_are_whole_graph_replays_of_enough_time():
    from tensor_partial_sum_gb300 import workloads as W
    small, big = W.WORKLOADS["tp_small"], W.WORKLOADS["f16_edges"]
    k = bench.config_steps(small, 20, 64)
    assert k % 64 == 0 and k * (small.bytes_per_call / 6.8e12 + 1e-6) > 1.9e-3  # about 2 ms of launches
    assert bench.config_steps(big, 20, 20) == 20
    assert bench.config_steps(big, 25, 20) == 40


def test_roofline_record_has_measured_and_nominal_fractions():
    from tensor_partial_sum_gb300 import workloads as W
    w = W.WORKLOADS["prefill"]
    r = bench.roofline(w, 20e-6)
    assert r["achieved"] == round(w.bytes_per_call / 20e-6 / 1e9, 1)
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert abs(r["frac_nominal"] - r["achieved"] / 8000.0) < 1e-3 and r["nominal_peak"] == 8000.0
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["kernel_us"] == 20.0


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


def test_launch_mode_follows_the_library_environment(monkeypatch):
    monkeypatch.delenv("AR_PDL", raising=False)
    monkeypatch.delenv("AR_L2_PREFETCH", raising=False)
    assert bench.launch_mode().startswith("programmatic dependent launches, first wave prefetches")
    monkeypatch.setenv("AR_PDL", "0")
    monkeypatch.setenv("AR_L2_PREFETCH", "0")
    assert bench.launch_mode() == "plain launches, no L2 prefetch"
