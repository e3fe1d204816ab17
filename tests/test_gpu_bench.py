"""bench.py keeps its output contract on a GPU: one JSON line with every
key the benchmark driver reads, consistent with itself."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def test_bench_line_has_the_contract_keys():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "300", "--warmup", "5", "--e2e-steps", "3",
           "--cpu-seconds", "1", "--cpu-seconds-per-config", "0.5", "--sustain", "0.2"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
              "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 300 and d["warmup"] == 5 and d["gpu_launches"] == 300
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and "workload" in d["config"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert 0.5 < r["frac"] < 1.5  # a kernel doing the work, against a measured copy peak
    bytes_per_step = d["config"]["bytes_per_step"]
    assert abs(d["value"] - bytes_per_step / (d["ms_per_step"] * 1e-3) / 1e9) / d["value"] < 1e-3
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert d["dtype"] == "f32" and r["frac_nominal"] > 0 and r["nominal_peak"] == 8000.0
    # one record per workload the benchmark is specified on
    cfgs = d["configs"]
    assert [cfgs[n]["cfg"] for n in ("tp_small", "decode", "prefill", "bf16_t3", "f16_edges")] == [1, 2, 3, 4, 5]
    assert cfgs["prefill"]["roofline"] == r and cfgs["prefill"]["value"] == d["value"]
    for name, rec in cfgs.items():
        assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1, name
        assert rec["cpu_baseline"]["value"] > 0, name
        if name == "decode":
            assert 0 < rec["us_per_call"] < 5.0 and rec["cpu_baseline"]["unit"] == "µs/call"
            continue
        rr = rec["roofline"]
        assert abs(rr["frac"] - rr["achieved"] / rr["peak"]) < 1e-3 and rr["frac_nominal"] > 0, name
        assert abs(rr["achieved"] - rec["value"]) / rec["value"] < 1e-2, name
        assert rec["us_per_call"] > 0 and {"sm_mhz", "reasons"} <= set(rec["clocks"]), name
        if rec["class"] == "prefill":
            assert rr["frac"] > 0.8, (name, rr["frac"])  # the bar the benchmark is specified with
