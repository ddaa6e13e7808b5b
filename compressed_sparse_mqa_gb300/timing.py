"""Timing helpers: CUDA-event timing on a given stream, CUDA-graph capture of a
step sequence, and nvidia-smi clock sampling during a timed region."""
from __future__ import annotations

import json
import os
import statistics
import subprocess
import tempfile
import time

import torch

SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while active."""

    def __init__(self, device_index: int = 0, period_ms: int = 100):
        self.device_index = device_index
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}", f"--query-gpu={SMI_FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = []
        for i, n in enumerate(names):
            if any(r[5 + i].lower().startswith("active") for r in rows):
                reasons.append(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def capture_graph(fn, n_steps: int, stream: torch.cuda.Stream):
    """Capture fn(t) for t in range(n_steps) into one CUDA graph on `stream`."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for t in range(n_steps):
                fn(t)
    return g


def time_graph(g: torch.cuda.CUDAGraph, reps: int, stream: torch.cuda.Stream) -> float:
    """Milliseconds for `reps` back-to-back replays, CUDA events on `stream`."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


class L2Flush:
    """A device buffer of twice the L2 size; flush() overwrites it on a stream, which
    evicts whatever the L2 held (the write allocates every line)."""

    def __init__(self, device=None):
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.nbytes = 2 * l2
        self.buf = torch.empty(self.nbytes // 4, dtype=torch.int32, device=dev)
        self.n = 0

    def flush(self, stream: torch.cuda.Stream):
        with torch.cuda.stream(stream):
            self.n += 1
            self.buf.fill_(self.n)


def time_graph_samples(g: torch.cuda.CUDAGraph, samples: int, stream: torch.cuda.Stream,
                       flush: "L2Flush | None" = None, replays: int = 1) -> list:
    """Milliseconds of each of `samples` timed regions, each `replays` back-to-back
    replays of g, timed with CUDA events on `stream`.  With `flush`, the L2 is
    overwritten on the same stream before each region and outside it; the flush also
    keeps the GPU busy while the host enqueues the region, so no launch gap is timed."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(samples)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for a, b in evs:
            if flush is not None:
                flush.flush(stream)
            a.record(stream)
            for _ in range(replays):
                g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def spread(ms: list) -> dict:
    """Median and spread of a list of sample times (ms)."""
    xs = sorted(ms)
    n = len(xs)

    def q(f):
        return xs[min(n - 1, max(0, int(round(f * (n - 1)))))]
    return {"median": statistics.median(xs), "min": xs[0], "p10": q(0.1), "p90": q(0.9), "max": xs[-1], "n": n}


def time_each(fn, n: int, stream: torch.cuda.Stream) -> float:
    """Average milliseconds of fn(t) over n calls, each bracketed by events on `stream`."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for t in range(n):
            evs[t][0].record(stream)
            fn(t)
            evs[t][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / n


def load_peaks(root: str) -> tuple[dict, str]:
    path = os.path.join(root, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"
