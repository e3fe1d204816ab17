#!/usr/bin/env python
"""Benchmark of the partial-sum reduction on GB300.

One step = one ar_reduce call over one batch of the workload (every step of
the hot path: load R partials, round each through the wire type, fold in
float, cast back, store to every destination).  Headline workload: prefill,
R=2 f32[2048,4096], bf16 wire, 2 destinations (128 MiB moved per call).

The same line carries a record per workload the benchmark is specified on
(``configs``): the small R=2 f32[32,4096] call, the decode-sized calls
(µs/call, CUDA-graph launched), prefill, R=4 bf16[4096,8192] and R=8
f32[8192,8192]; each with its roofline fraction and the oracle timed on the
host cores beside it.

Prints ONE JSON line (rank 0).  Multi-GPU: launch under torchrun; every rank
runs the same independent reduction on its own GPU (weak scaling, no
collective on the data path); timing is the max over ranks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import datetime as dt
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s (% of roofline) prefill-size; µs/call decode-size"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
# the HBM3e bandwidth the roofline is usually quoted against (GB300, ~8 TB/s)
NOMINAL_HBM_GBS = 8000.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# the file that defines the timed kernel (ar_reduce_kernel) and its helpers, and the table
# of its instantiations: a launch's traffic depends on this code, not on the rest of the
# host code or the other kernels
KERNEL_SOURCES = [os.path.join(ROOT, "tensor_partial_sum_gb300", "csrc", f)
                  for f in ("ar_kernels.cuh", "ar_dispatch.h")]
# GPU clock cycles of idle work enqueued ahead of the start event (about 0.2 ms)
LEAD_CYCLES = 400_000
# the workloads the benchmark is specified on, in their order, with the class each is judged as
CONFIGS = [("tp_small", 1, "small"), ("decode", 2, "decode"), ("prefill", 3, "prefill"),
           ("bf16_t3", 4, "prefill"), ("f16_edges", 5, "prefill")]


# ---- distributed plumbing (also exercised by the CPU tests with gloo) -------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if dist.get_backend() == "nccl":  # on this rank's own GPU, named so NCCL need not guess it
            import torch
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank moved bytes_per_step * steps bytes;
    the job took as long as its slowest rank."""
    return world * bytes_per_step * steps / max_seconds / 1e9


# ---- measured peaks, clocks, traffic -----------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def code_tokens(text: str) -> str:
    """Source text without comments and with whitespace collapsed: what the
    compiler sees, so editing a comment does not count as a kernel change."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def sources_digest() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p) as f:
            h.update(code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(workload: str, path: str = TRAFFIC_FILE):
    """DRAM bytes per launch of the workload's kernel from the committed ncu
    counters, or None when the file has no entry for the workload or the
    kernel sources changed since the counters were taken."""
    try:
        with open(path) as f:
            e = json.load(f)["workloads"][workload]
        if e["source_digest"] != sources_digest():
            return None
        return int(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


def roofline(w, kernel_s: float) -> dict:
    """The roofline record of one workload: algorithmic bytes per launch over
    the average launch time, against the measured copy peak and the nominal
    HBM3e figure."""
    peak, peak_src = hbm_peak()
    achieved = w.bytes_per_call / kernel_s / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic_per_launch(w.name), "peak_source": peak_src,
            "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "nominal_peak": NOMINAL_HBM_GBS,
            "kernel_us": round(kernel_s * 1e6, 3)}


class ClockSampler:
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        rows = []
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 9:
                continue
            try:
                ts = dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append({"t": ts, "sm": float(parts[1]), "max": float(parts[2]),
                             "reasons": [n for n, v in zip(self.REASONS, parts[5:]) if v == "Active"]})
            except ValueError:
                continue
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        inside = [r for r in rows if t0 <= r["t"] <= t1]
        window = "timed region"
        if len(inside) < 3:
            inside, window = rows, "sustained pre-run and timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
        reasons = sorted({x for r in inside for x in r["reasons"]})
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["max"] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def throttled(clocks) -> bool:
    """True when the clock samples show a slowdown that invalidates a timing
    (sw_power_cap alone does not)."""
    return any(r in REJECT_REASONS for r in clocks.get("reasons", []))


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
    except Exception:  # pragma: no cover - older torch
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[device_index] if vis else str(device_index)


def launch_mode() -> str:
    """How the library launches its kernels, from the environment it reads at ar_init."""
    pdl = os.environ.get("AR_PDL", "1") != "0"
    pf = os.environ.get("AR_L2_PREFETCH", "1") != "0"
    return ("programmatic dependent launches" if pdl else "plain launches") + \
        (", first wave prefetches its sources into L2 before the wait" if pf else ", no L2 prefetch")


def config_steps(w, steps: int, group: int, min_seconds: float = 2e-3) -> int:
    """Timed launches for a workload measured beside the headline: at least
    ``steps``, enough for about ``min_seconds`` of GPU time at the HBM peak
    (so a microsecond-sized call is not timed on a handful of launches), and
    a whole number of replays of its ``group``-launch graph (no eager
    launches inside the timed region)."""
    peak, _ = hbm_peak()
    est = w.bytes_per_call / (peak * 1e9) + 1e-6
    want = max(steps, math.ceil(min_seconds / est))
    return group * math.ceil(want / group)


# ---- the oracle as CPU baseline ------------------------------------------------

def oracle_step(w, srcs, r0: int, r1: int):
    """The oracle's version of one step over rows [r0, r1) (its results are
    new arrays; the call releases the GIL while the C oracle runs)."""
    import oracle
    a, b = r0 * w.ne0, r1 * w.ne0
    if w.op == "pack":
        return oracle.wire_pack(srcs[0][a:b], w.dst, w.wire)
    if w.op == "reduce":
        return oracle.reduce([s[a:b] for s in srcs[:w.R]], w.n_dsts, w.dst, w.wire)
    res, res_stride = None, None
    if w.residual == "full":
        res = srcs[w.R][a:b]
    elif w.residual == "row":
        res, res_stride = srcs[w.R], 0
    holes = [None if r in w.inactive else s[a:b] for r, s in enumerate(srcs[:w.R])]
    return oracle.reduce_2d(holes, w.n_dsts, w.dst, w.wire, w.ne0, r1 - r0, inactive=w.inactive, residual=res,
                            residual_stride=res_stride)


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rate(srcs, w, seconds: float, steps: int = 0, threads: int = 1):
    """Time the oracle, as it stands, on a sample of whole rows of the
    workload; with threads > 1 each pass splits the sample into contiguous
    row ranges, one per thread (every element is independent, so the bytes
    are those of one call).  With steps == 0 the sample and repetitions are
    sized to take about `seconds`; otherwise `steps` repetitions of a sample
    sized to take about seconds / steps each.  Returns (GB/s, elapsed,
    sample text)."""
    from concurrent.futures import ThreadPoolExecutor

    def one_pass(pool, rows, nt):
        cuts = [rows * k // nt for k in range(nt + 1)]
        list(pool.map(lambda k: oracle_step(w, srcs, cuts[k], cuts[k + 1]), range(nt)))

    with ThreadPoolExecutor(threads) as pool:
        # a pass costs about a + b * rows: fit a and b on two probe passes
        r1 = max(1, min(w.ne1, threads))
        r2 = max(r1 + 1, min(w.ne1, max(8 * threads, (1 << 18) // w.ne0)))
        cost = []
        for r in (r1, r2):
            t = time.perf_counter()
            one_pass(pool, r, min(threads, r))
            cost.append(time.perf_counter() - t)
        b = max((cost[1] - cost[0]) / (r2 - r1), 1e-9)
        a = max(cost[0] - b * r1, 0.0)
        budget = seconds / steps if steps else seconds
        rows = int(min(w.ne1, max(1, (budget - a) / b)))
        # at least one row per thread, so that every core works in every pass
        # (a pass then costs a + b * threads, which may exceed a tiny budget)
        rows = max(rows, min(threads, w.ne1))
        per_pass = a + b * rows
        reps = steps if steps else max(1, int(seconds / per_pass))
        nt = max(1, min(threads, rows))
        t = time.perf_counter()
        for _ in range(reps):
            one_pass(pool, rows, nt)
        el = time.perf_counter() - t
    moved = w.bytes_per_call * rows / w.ne1 * reps
    return (moved / el / 1e9, el,
            f"first {rows} of {w.ne1} rows ({rows * w.ne0} of {w.nelem} elements) of the workload, "
            f"{reps} pass(es) on {nt} thread(s), {el:.1f} s")


def oracle_decode_rate(w, seconds: float, threads: int, calls: int = 256):
    """Decode-sized calls through the oracle on ``threads`` host cores, each
    thread running whole calls (of the first ``calls`` per-call inputs, in
    turn) for about ``seconds``.  Returns (µs per call for all threads
    together, elapsed, sample text)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from tensor_partial_sum_gb300 import workloads as W
    inputs = [W.generate(w, call=k) for k in range(min(calls, w.calls))]

    def worker(t):
        n, t_end = 0, time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            oracle.reduce(inputs[(t + n * threads) % len(inputs)], w.n_dsts, w.dst, w.wire)
            n += 1
        return n

    start = time.perf_counter()
    with ThreadPoolExecutor(threads) as pool:
        done = sum(pool.map(worker, range(threads)))
    el = time.perf_counter() - start
    return (el * 1e6 / done, el,
            f"{done} whole calls (first {len(inputs)} of {w.calls} per-call inputs, cycled) on {threads} "
            f"thread(s), {el:.1f} s")


def cpu_baseline_record(w, srcs, seconds: float, single_seconds: float = 0.0) -> dict:
    """The oracle on every host core (and, when ``single_seconds``, on one)."""
    nt = host_threads()
    if w.calls > 1:
        us, _, sample = oracle_decode_rate(w, seconds, nt)
        return {"value": round(us, 3), "unit": "µs/call", "cores": nt, "kind": "oracle", "sample": sample,
                "machine": platform.machine()}
    v, _, sample = oracle_rate(srcs, w, seconds, threads=nt)
    rec = {"value": round(v, 4), "unit": UNIT, "cores": nt, "kind": "oracle", "sample": sample,
           "machine": platform.machine()}
    if single_seconds > 0:
        v1, _, sample1 = oracle_rate(srcs, w, single_seconds)
        rec["single_thread"] = {"value": round(v1, 4), "sample": sample1}
    return rec


# ---- our arm -----------------------------------------------------------------

class Runner:
    """Device, stream and clock sampler shared by every workload measured in
    one run."""

    def __init__(self, args):
        import torch

        from tensor_partial_sum_gb300 import build as lib_build
        self.args = args
        self.rank, self.local_rank, self.world = dist_env()
        torch.cuda.set_device(self.local_rank)
        self.dev = torch.device("cuda", self.local_rank)
        dist_init(self.world, "nccl")
        if lib_build.stale():
            if self.rank == 0:
                lib_build.build()
            barrier()
        props = torch.cuda.get_device_properties(self.dev)
        self.l2 = getattr(props, "L2_cache_size", 129 * 1000 * 1000) or 129 * 1000 * 1000
        self.sampler = ClockSampler(gpu_id_for(self.local_rank))
        self.stream = torch.cuda.Stream(self.dev)

    def measure(self, w, srcs_np, steps: int, exact_steps: bool, keep: bool = False):
        """Time ``steps`` calls of workload ``w`` (graph-launched, back to
        back, rotating buffer sets so every step's inputs come from HBM).
        With ``exact_steps`` False the count is rounded up to whole graph
        replays.  Returns a dict of timings and launch facts."""
        import numpy as np
        import torch

        import tensor_partial_sum_gb300 as tps
        args, dev, stream = self.args, self.dev, self.stream
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dst]

        def dev_tensor(a):
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
            return t.to(dev).view(tdt)

        # rotating buffer sets: each step's inputs were last touched sets-1 steps ago
        nsets = 1 if w.bytes_per_call >= 3 * self.l2 else math.ceil(3 * self.l2 / w.bytes_per_call)
        ne0, ne1, pad = w.ne0, w.ne1, w.row_pad

        def rows_tensor(a=None):
            """A device tensor of ne1 rows at a row stride of ne0 + pad elements."""
            t = torch.empty((ne1, ne0 + pad), dtype=tdt, device=dev)
            if pad:
                t[:, ne0:].fill_(0)
            if a is not None:
                t[:, :ne0].copy_(dev_tensor(a).view(ne1, ne0))
            return t

        base_src = [dev_tensor(a) if pad == 0 else rows_tensor(a) for a in srcs_np[:w.R]]
        residual_base = dev_tensor(srcs_np[w.R]) if w.residual else None
        sets = []
        for k in range(nsets):
            s = base_src if k == 0 else [b.clone() for b in base_src]
            if w.op == "pack":
                d = [torch.empty(w.nelem, dtype={"f32": torch.float32, "f16": torch.float16,
                                                 "bf16": torch.bfloat16}[w.wire], device=dev)]
            else:
                d = [torch.empty(w.nelem, dtype=tdt, device=dev) if pad == 0 else rows_tensor()
                     for _ in range(w.n_dsts)]
            res = None if residual_base is None else (residual_base if k == 0 else residual_base.clone())
            sets.append((s, d, res))
        tps.ar_init(w.R, w.nelem)
        if args.bw_blocks_per_sm:
            tps.ar_set_option("bw_blocks_per_sm", args.bw_blocks_per_sm)
        if args.variant != "auto":
            tps.ar_set_option("forced_variant", tps.ar.VARIANTS[args.variant])
        es = w.elem_bytes
        layouts = []
        for s, d, res in sets:
            if w.op != "reduce_ex":
                layouts.append(None)
                continue
            layouts.append(tps.make_layout(
                ne0, ne1, src_row_bytes=[(ne0 + pad) * es] * w.R, dst_row_bytes=[(ne0 + pad) * es] * w.n_dsts,
                residual=res, residual_row_bytes=0 if w.residual == "row" else None, inactive=w.inactive))
            for r in w.inactive:
                s[r] = None

        def step(i):
            k = i % nsets
            s, d, res = sets[k]
            if w.op == "reduce":
                tps.ar_reduce(s, d, nelem=w.nelem, dst_dtype=w.dst, wire_dtype=w.wire, stream=stream)
            elif w.op == "reduce_ex":
                tps.ar_reduce_ex(s, d, layouts[k], w.dst, w.wire, stream=stream)
            else:
                tps.ar_wire_pack(s[0], d[0], nelem=w.nelem, dst_dtype=w.dst, wire_dtype=w.wire, stream=stream)

        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                step(i)
        torch.cuda.synchronize(dev)
        variant = ({v: k for k, v in tps.ar.VARIANTS.items()}[tps.ar_query("last_variant")]
                   if w.op == "reduce" else w.op)

        # graph of G steps, replayed back to back in the timed region
        G = max(1, min(steps, nsets * max(1, math.ceil(64 / nsets))))
        if not exact_steps:
            steps = G * math.ceil(steps / G)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(G):
                step(i)
        replays, rem = divmod(steps, G)

        def timed_region():
            """Sustained pre-run, then exactly `steps` steps between events;
            clocks are sampled throughout.  Returns (seconds, clocks)."""
            self.sampler.start()
            with torch.cuda.stream(stream):  # sustained pre-run so clocks are sampled under load
                t_end = time.perf_counter() + args.sustain
                while time.perf_counter() < t_end:
                    graph.replay()
                    torch.cuda.synchronize(dev)
            barrier()
            torch.cuda.synchronize(dev)
            t0 = dt.datetime.now()
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                # keep the GPU busy while the host submits the timed launches, so that
                # the host's submission latency does not sit between the start event
                # and the first launch (the device time of the K steps is measured)
                torch.cuda._sleep(LEAD_CYCLES)
                start.record(stream)
                for _ in range(replays):
                    graph.replay()
                for i in range(rem):
                    step(i)
                end.record(stream)
            torch.cuda.synchronize(dev)
            t1 = dt.datetime.now()
            barrier()
            return start.elapsed_time(end) / 1e3, ClockSampler.summarize(self.sampler.stop(), t0, t1)

        elapsed, clocks = timed_region()
        if throttled(clocks):  # a slowed-down GPU: measure once more and keep the second run
            first = clocks
            elapsed, clocks = timed_region()
            clocks["remeasured_after"] = first["reasons"]
        # for context: launches bracketed one by one by event pairs
        pairs = []
        with torch.cuda.stream(stream):
            for i in range(min(steps, 100)):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                step(i)
                b.record(stream)
                pairs.append((a, b))
        torch.cuda.synchronize(dev)
        m = {"elapsed": elapsed, "max_elapsed": max_over_ranks(elapsed, dev), "steps": steps, "clocks": clocks,
             "variant": variant, "kernel_pair_us": statistics.median(a.elapsed_time(b) for a, b in pairs) * 1e3,
             "l2": f"{nsets} rotating buffer sets ({nsets * w.bytes_per_call / 2**20:.0f} MiB) cycled, "
                   f"L2 {self.l2 / 2**20:.0f} MiB: each step's inputs were last touched {nsets - 1} steps earlier"
                   if nsets > 1 else f"inputs {w.bytes_per_call / 2**20:.0f} MiB > 3x L2",
             "timing": f"CUDA graph of {G} launches replayed {replays}x (+{rem} eager), "
                       "CUDA events on the launching stream, the start event queued behind ~0.2 ms of "
                       "idle GPU work so the host's submission is not timed"}
        del graph
        if keep:
            m["sets"] = sets
        else:
            del sets, base_src, residual_base
            torch.cuda.empty_cache()
        tps.ar_free()
        return m

    def e2e(self, w, srcs_np, sets):
        """End to end through the host entry point: pinned host partials in,
        pinned host results out, every step inside the timed region."""
        import numpy as np
        import torch

        import tensor_partial_sum_gb300 as tps
        args, dev, stream = self.args, self.dev, self.stream
        tps.ar_init(w.R, w.nelem)
        h_srcs = [torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory() for a in srcs_np]
        h_dsts = [torch.empty(w.nelem, dtype=h_srcs[0].dtype).pin_memory() for _ in range(w.n_dsts)]
        d_srcs, d_dsts, _ = sets[0]

        def e2e_time(staged: bool) -> float:
            def one():
                tps.ar_reduce_host(h_srcs, h_dsts, d_srcs if staged else None, d_dsts if staged else None,
                                   nelem=w.nelem, dst_dtype=w.dst, wire_dtype=w.wire, stream=stream)
            for _ in range(3):
                one()
            torch.cuda.synchronize(dev)
            barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.e2e_steps):
                one()
            b.record(stream)
            torch.cuda.synchronize(dev)
            return max_over_ranks(a.elapsed_time(b) / 1e3, dev)

        direct = e2e_time(staged=False)
        staged = e2e_time(staged=True)
        tps.ar_free()
        return {"value": round(aggregate_gbs(w.bytes_per_call, args.e2e_steps, self.world, direct), 2),
                "unit": UNIT, "h2d_bytes_per_step": w.R * w.nelem * w.elem_bytes,
                "d2h_bytes_per_step": w.n_dsts * w.nelem * w.elem_bytes, "steps": args.e2e_steps,
                "call": "ar_reduce_host without staging: the kernel loads the pinned host partials and "
                        "stores the pinned host results over NVLink-C2C",
                "staged_pipeline_value": round(aggregate_gbs(w.bytes_per_call, args.e2e_steps, self.world,
                                                             staged), 2),
                "staged_pipeline_call": "ar_reduce_host with device staging: chunked H2D copy, kernel, "
                                        "D2H copy on three streams"}


def run_ours(args):
    import torch

    from tensor_partial_sum_gb300 import workloads as W

    run = Runner(args)
    w = W.WORKLOADS[args.workload]
    srcs_np = W.generate(w)
    m = run.measure(w, srcs_np, args.steps, exact_steps=True, keep=w.op == "reduce" and args.e2e_steps > 0)
    value = aggregate_gbs(w.bytes_per_call, args.steps, run.world, m["max_elapsed"])
    # average launch duration over the timed region: the launches run back to
    # back, so this includes the gaps between them (a conservative figure)
    kernel_s = m["elapsed"] / args.steps
    roof = roofline(w, kernel_s)
    roof["kernel_us_event_pairs"] = round(m["kernel_pair_us"], 3)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": run.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["max_elapsed"] * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dst,
        "accumulate": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.describe()}", "bytes_per_step": w.bytes_per_call,
                   "variant": m["variant"], "parallelism": f"{run.world} independent replica(s), no collective",
                   "l2": m["l2"], "timing": m["timing"], "launch": launch_mode()},
        "roofline": roof,
        "gpu_launches": args.steps,
        "clocks": m["clocks"],
    }
    if "sets" in m:
        result["e2e"] = run.e2e(w, srcs_np, m.pop("sets"))
        torch.cuda.empty_cache()
    cpu_on = run.rank == 0 and run.world == 1 and args.cpu_seconds > 0
    if cpu_on:
        # the oracle on every host core, and on one for reference
        result["cpu_baseline"] = cpu_baseline_record(w, srcs_np, args.cpu_seconds / 2, args.cpu_seconds / 2)
    headline = {"cfg": dict((n, c) for n, c, _ in CONFIGS).get(w.name), "workload": f"{w.name}: {w.describe()}",
                "value": result["value"], "unit": UNIT, "us_per_call": round(kernel_s * 1e6, 3),
                "variant": m["variant"], "steps": args.steps, "roofline": roof, "clocks": m["clocks"],
                "timing": m["timing"], "l2": m["l2"], "measured_as": "the headline (value) of this line"}
    if "cpu_baseline" in result:
        headline["cpu_baseline"] = result["cpu_baseline"]
    del srcs_np

    # every workload the benchmark is specified on, one record each
    wanted = [c for c in CONFIGS if args.configs == "all" or c[0] in args.configs.split(",")]
    records = {}
    for name, cfg, klass in wanted:
        cw = W.WORKLOADS[name]
        if name == w.name:
            records[name] = dict(headline, cfg=cfg, **{"class": klass})
            continue
        if cw.calls > 1:
            rec = bench_decode(run.dev, run.stream)
            rec.update(cfg=cfg, **{"class": klass})
            if cpu_on:
                rec["cpu_baseline"] = cpu_baseline_record(cw, None, args.cpu_seconds_per_config)
            records[name] = rec
            continue
        csrcs = W.generate(cw)
        cm = run.measure(cw, csrcs, config_steps(cw, args.steps, 1), exact_steps=False)
        ks = cm["elapsed"] / cm["steps"]
        rec = {"cfg": cfg, "class": klass, "workload": f"{cw.name}: {cw.describe()}",
               "value": round(aggregate_gbs(cw.bytes_per_call, cm["steps"], run.world, cm["max_elapsed"]), 2),
               "unit": UNIT, "us_per_call": round(ks * 1e6, 3), "variant": cm["variant"], "steps": cm["steps"],
               "bytes_per_call": cw.bytes_per_call, "roofline": dict(roofline(cw, ks),
                                                                     kernel_us_event_pairs=round(cm["kernel_pair_us"], 3)),
               "clocks": cm["clocks"], "timing": cm["timing"], "l2": cm["l2"]}
        if cpu_on:
            rec["cpu_baseline"] = cpu_baseline_record(cw, csrcs, args.cpu_seconds_per_config)
        del csrcs
        records[name] = rec
    if records:
        result["configs"] = records
    if run.rank == 0:
        print(json.dumps(result), flush=True)


def bench_decode(dev, stream):
    """Decode-sized calls: R=4 f32[1,4099], f16 wire, 4 destinations, 10000
    calls with their own buffers and per-call seeds, captured in one CUDA
    graph; microseconds per call = graph replay time / calls."""
    import numpy as np
    import torch

    import tensor_partial_sum_gb300 as tps
    from tensor_partial_sum_gb300 import workloads as W

    w = W.WORKLOADS["decode"]
    row = (w.nelem + 3) // 4 * 4  # pad rows to 16 bytes so every buffer is aligned
    buf = torch.zeros((w.calls, w.R + w.n_dsts, row), dtype=torch.float32, device=dev)
    host = np.zeros((w.calls, w.R, w.nelem), dtype=np.float32)
    for k in range(w.calls):
        host[k] = np.stack(W.generate(w, call=k))
    buf[:, :w.R, :w.nelem].copy_(torch.from_numpy(host))
    del host
    tps.ar_init(w.R, w.nelem)
    ptr = buf.data_ptr()
    stride_call, stride_buf = buf.stride(0) * 4, buf.stride(1) * 4
    calls = [([ptr + k * stride_call + r * stride_buf for r in range(w.R)],
              [ptr + k * stride_call + (w.R + d) * stride_buf for d in range(w.n_dsts)]) for k in range(w.calls)]

    def one(k):
        s, d = calls[k]
        tps.ar_reduce(s, d, nelem=w.nelem, dst_dtype="f32", wire_dtype=w.wire, stream=stream)

    with torch.cuda.stream(stream):
        for k in range(min(100, w.calls)):
            one(k)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for k in range(w.calls):
            one(k)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    with torch.cuda.stream(stream):
        graph.replay()
        for _ in range(5):
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b) * 1e3 / w.calls)
        a.record(stream)
        for k in range(w.calls):
            one(k)
        b.record(stream)
    torch.cuda.synchronize(dev)
    eager = a.elapsed_time(b) * 1e3 / w.calls
    # the same calls through prepared calls (buffer checks and pointer arrays done once)
    prepared = [tps.PreparedReduce(s, d, nelem=w.nelem, dst_dtype="f32", wire_dtype=w.wire, stream=stream)
                for s, d in calls]
    with torch.cuda.stream(stream):
        for k in range(min(100, w.calls)):
            prepared[k]()
        torch.cuda.synchronize(dev)
        a.record(stream)
        for k in range(w.calls):
            prepared[k]()
        b.record(stream)
    torch.cuda.synchronize(dev)
    eager_prepared = a.elapsed_time(b) * 1e3 / w.calls
    variant = {v: k for k, v in tps.ar.VARIANTS.items()}[tps.ar_query("last_variant")]
    del graph, buf
    tps.ar_free()
    torch.cuda.empty_cache()
    us = statistics.median(times)
    return {"us_per_call": round(us, 3), "unit": "µs/call", "target_us": 5.0,
            "workload": f"{w.name}: {w.describe()}", "variant": variant,
            "timing": f"one CUDA graph of {w.calls} ar_reduce nodes, median of 5 replays",
            "us_per_call_eager_stream": round(eager, 3),
            "us_per_call_eager_prepared": round(eager_prepared, 3),
            "bytes_per_call": w.bytes_per_call,
            "gbs": round(w.bytes_per_call / (us * 1e-6) / 1e9, 2)}


# ---- reference arm: the oracle on the host cores ------------------------------

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    from tensor_partial_sum_gb300 import workloads as W

    w = W.WORKLOADS[args.workload]
    srcs = W.generate(w)
    budget = args.ref_seconds
    nt = host_threads()
    # untimed warm-up passes on a small sample, then the timed steps, on every host core
    oracle_rate(srcs, w, min(1.0, budget / 10), steps=args.warmup, threads=nt)
    value, el, text = oracle_rate(srcs, w, budget, steps=args.steps, threads=nt)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dst, "accumulate": "f32",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.describe()}", "bytes_per_step": w.bytes_per_call,
                   "variant": "oracle (scalar C, element by element)",
                   "parallelism": "oracle on rank 0 only, contiguous row ranges on every host core",
                   "l2": "host caches; each step is a bounded sample of the workload's rows",
                   "timing": "wall clock (time.perf_counter) around the timed steps",
                   "launch": "none: the oracle runs on the host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": nt, "kind": "oracle", "sample": text,
                         "machine": platform.machine()},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="prefill", help="the headline workload (value, roofline)")
    p.add_argument("--configs", default="all",
                   help="workloads measured beside the headline: all, none, or names separated by commas")
    p.add_argument("--e2e-steps", type=int, default=100)
    p.add_argument("--sustain", type=float, default=1.0, help="seconds of untimed load before timing")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle seconds for the headline workload")
    p.add_argument("--cpu-seconds-per-config", type=float, default=3.0,
                   help="oracle seconds for each other workload")
    p.add_argument("--ref-seconds", type=float, default=60.0)
    p.add_argument("--variant", default="auto", help="force a kernel variant of ar_reduce (auto, bandwidth, tma, ...)")
    p.add_argument("--bw-blocks-per-sm", type=int, default=0,
                   help="0: bandwidth grid covers the tensor; n: persistent grid of n CTAs per SM")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.steps < 1:
        p.error("--steps must be at least 1")
    world = dist_env()[2]
    if args.gpus != world:
        p.error(f"--gpus {args.gpus} but {world} process(es): for N > 1 launch one process per GPU "
                f"(python -m torch.distributed.run --nproc-per-node N ... bench.py --gpus N)")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
