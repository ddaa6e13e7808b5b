#!/usr/bin/env python3
"""Benchmark of the compressed sparse MQA attention path on one GB300.

Headline step: one batch-1 decode token through one ratio-4 layer with the
indexer at context 32768 (8192 compressed rows, top-512, 128-row raw window, 64
heads, head_dim 128, fp16): ds4a_indexer_topk_compress (the indexer query and
the compressor's update for the new token, in one launch) -> ds4a_attn_decode.
Metric: tokens/s/layer (= steps/s) and the HBM bandwidth the step's algorithmic
bytes imply.

Inputs are resident in HBM.  The timed steps rotate over enough independent
copies of the layer state that the working set is more than twice the L2, so
each step streams its keys from DRAM.  The timed region is a CUDA graph of
the steps, replayed back to back, timed with CUDA events on its stream.

Printed (one JSON line on rank 0): the headline metric, e2e (the same step
through the Python binding with the step's inputs copied from pinned host
memory and the output read back, every step), the roofline of the dominant
kernel, the oracle's CPU time, the clocks seen, and sub-results for the ratio-128
decode layer, the 2048-token prefill chunk and the 43-layer decode stack.
`--impl reference` times the fp64 CPU oracle on the same step instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn tokens/s/layer & HBM GB/s (% of peak); prefill tokens/s (% tensor peak)"
UNIT = "tokens/s/layer"
# algorithmic flops of the prefill chunk: causal indexer GEMM + attention over 640 rows per query
C4_FLOPS = 47.11e9


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=65536)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sub", action="store_true", help="skip the C3/C4/C5 sub-results")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", choices=["c3", "c4", "c5"], default=None,
                    help="run one sub-configuration alone and print its result (for profiling)")
    return ap.parse_args()


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ms: float, steps: int, world: int) -> tuple[float, float]:
    """The slowest rank's time (ms) for `steps` steps on every rank, and the whole-job
    rate world * steps / that time (steps per second over all ranks)."""
    ms = max_over_ranks(ms, world)
    return ms, world * steps / (ms / 1e3)


def graph_size(k: int, cap: int = 1024) -> int:
    if k <= cap:
        return k
    for g in range(cap, 0, -1):
        if k % g == 0:
            return g
    return 1


def rotation_copies(bytes_per_copy: int, l2_bytes: int, minimum: int = 2) -> int:
    return max(minimum, math.ceil(2 * l2_bytes / max(bytes_per_copy, 1)) + 1)


KERNEL_SOURCES = {"indexer_topk_compress": ["indexer.cu", "compress_dev.cuh", "select.cuh"],
                  "attn_decode": ["attention.cu"]}


def kernel_traffic(name: str):
    """DRAM bytes per launch from the committed ncu capture of this kernel, or None
    when the kernel's source has changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    srcs = [os.path.join(ROOT, "compressed_sparse_mqa_gb300", "csrc", f) for f in KERNEL_SOURCES.get(name, [])]
    if not os.path.exists(path) or not srcs or not all(os.path.isfile(f) for f in srcs):
        return None
    with open(path) as f:
        entry = json.load(f).get(name)
    if not entry:
        return None
    return entry["dram_bytes_per_launch"] if entry.get("source_sha256") == source_digest(srcs) else None


def source_digest(paths) -> str:
    """sha256 over the concatenated contents of a kernel's source files."""
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------

def time_decode_rotation(layers, steps, warmup, stream):
    """Graph-replay timing of `steps` decode steps rotating over `layers`.  Returns ms total."""
    from compressed_sparse_mqa_gb300 import timing
    R = len(layers)
    G = graph_size(steps)
    gw = timing.capture_graph(lambda t: layers[t % R].step(), max(1, min(warmup, 1024)), stream)
    g = timing.capture_graph(lambda t: layers[t % R].step(), G, stream)
    for _ in range(max(1, math.ceil(warmup / max(1, min(warmup, 1024))))):
        gw.replay()
    import torch
    torch.cuda.synchronize()
    return g, G


def run_ours(args, rank, world, local):
    import torch

    from compressed_sparse_mqa_gb300 import configs, ds4a, timing
    from compressed_sparse_mqa_gb300.layer import DecodeLayer, PrefillLayer

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA library is the only implementation)")
    torch.cuda.set_device(local)
    ds4a.lib()   # raises if the library is not built
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    peaks, peak_src = timing.load_peaks(ROOT)
    hbm_peak = float(peaks["hbm_gbs"])
    stream = torch.cuda.Stream()
    if args.only:
        fn = {"c3": lambda: sub_decode(configs.C3, l2, stream, hbm_peak),
              "c4": lambda: sub_prefill(configs.C4, l2, stream, peaks),
              "c5": lambda: sub_stack(l2, stream, hbm_peak)}[args.only]
        return {"only": args.only, "result": fn()}

    # ---- headline: C2 decode step --------------------------------------------------------
    inst = configs.decode(configs.C2)
    base = DecodeLayer(inst)
    step_bytes = base.bytes_touched()
    R = rotation_copies(step_bytes, l2, minimum=8)
    layers = [base] + [base.clone() for _ in range(R - 1)]
    with torch.cuda.stream(stream):
        for L in layers[:4]:
            L.step()
    torch.cuda.synchronize()
    g, G = time_decode_rotation(layers, args.steps, args.warmup, stream)
    reps = args.steps // G
    barrier(world)
    with timing.ClockSampler(local) as clk:
        ms = timing.time_graph(g, reps, stream)
    barrier(world)
    clocks = clk.summary()
    steps = G * reps
    ms, value = job_throughput(ms, steps, world)
    s_per_step = ms / 1e3 / steps
    gbs = step_bytes / s_per_step / 1e9

    # ---- per-kernel durations (events around each launch, on the launching stream) -------
    def k_prep(t):
        L = layers[t % R]
        ds4a.ds4a_indexer_topk_compress(L.q_idx, L.kidx, L.p, L.ratio, L.topk, L.sel, L.sel_n, L.ws,
                                        L.ring_k[L.slot:L.slot + 1], L.ring_v[L.slot:L.slot + 1], L.w, L.state,
                                        L.comp_k, L.comp_v)

    def k_attn(t):
        L = layers[t % R]
        ds4a.ds4a_attn_decode(L.q, L.ring_k[:L.n_win], L.ring_v[:L.n_win], L.comp_k, L.comp_v, L.sel, L.topk,
                              L.scale, L.out)

    # each kernel alone: a CUDA graph of n_k back-to-back launches over the rotation,
    # CUDA events around its replays on the launching stream; average per launch
    n_k = 1024
    kt = {}
    for name, fn in [("indexer_topk_compress", k_prep), ("attn_decode", k_attn)]:
        gk = timing.capture_graph(fn, n_k, stream)
        gk.replay()
        kt[name] = timing.time_graph(gk, 4, stream) / (4 * n_k)
    D, H = base.D, base.H
    kbytes = {
        # indexer keys + query + kept indices, and the compressor's token, score vector and state
        "indexer_topk_compress": base.n_vis * base.kidx.shape[1] * 2 + base.kidx.shape[1] * 2 + base.topk * 4 + 4
        + 2 * D * 2 + D * 4 + (2 + 2 * D) * 4,
        "attn_decode": 2 * H * D * 2 + 2 * (base.n_win + base.topk) * D * 2 + base.topk * 4,
    }
    launches_per_step = len(kt)   # the kernels of one step, each timed above
    dom = max(kt, key=kt.get)
    achieved = kbytes[dom] / (kt[dom] / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": kernel_traffic(dom),
                "peak_source": f"{peak_src} hbm_gbs",
                "kernel_us": {k: round(v * 1e3, 3) for k, v in kt.items()},
                "kernel_bytes": kbytes}

    # ---- e2e: per-step inputs from pinned host memory, output read back every step ----------
    e2e = run_e2e(layers, stream, n_steps=min(2000, max(200, args.steps // 32)))

    # ---- sub-results ---------------------------------------------------------------------------
    sub = {}
    if not args.no_sub:
        sub["c3_decode_ratio128_ctx131072"] = sub_decode(configs.C3, l2, stream, hbm_peak)
        sub["c4_prefill_2048_ratio4"] = sub_prefill(configs.C4, l2, stream, peaks)
        sub["c5_stack_43_layers_ctx65536"] = sub_stack(l2, stream, hbm_peak)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms / steps, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 (fp32 accumulate)",
        "data": "synthetic (seeded SplitMix64/Box-Muller, N(0,1) values)",
        "config": {"workload": "C2 batch-1 decode, ratio-4 layer + indexer top-512, ctx 32768",
                   "heads": H, "kv_heads": 1, "head_dim": D, "window": base.W, "compressed_rows": base.n_vis,
                   "topk": base.topk, "index_dim": base.kidx.shape[1],
                   "l2_policy": f"rotate {R} layer copies ({R * step_bytes / 1e6:.0f} MB touched > 2x L2 "
                                f"{l2 / 1e6:.0f} MB)",
                   "timed_region": f"CUDA graph of {G} steps x {reps} replays",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4), "bytes_per_step": step_bytes,
        "e2e": e2e, "gpu_launches": launches_per_step * steps, "roofline": roofline, "clocks": clocks,
        "sub": sub,
    }
    if rank == 0 and args.cpu_seconds > 0:
        line["cpu_baseline"] = cpu_baseline(inst, args.cpu_seconds)
    return line


def loaded_cudart():
    """The CUDA runtime library this process already has loaded (torch's), opened by
    its own path so that its streams are torch's; None if there is none to reuse."""
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            paths = [line.split()[-1] for line in f if "libcudart.so" in line]
    except OSError:
        return None
    if not paths:
        return None
    rt = ctypes.CDLL(paths[0])
    rt.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    rt.cudaStreamSynchronize.argtypes = [ctypes.c_void_p]
    return rt


def run_e2e(layers, stream, n_steps):
    """Steps through the public API with the step's inputs copied in from pinned host
    memory and the output read back, every step, on the host clock.  Each layer's
    step is marshalled once (DecodeLayer.bind); the copies are cudaMemcpyAsync calls
    on the step's stream (torch copies if the runtime library is not reachable)."""
    import torch

    from compressed_sparse_mqa_gb300 import ds4a
    R = len(layers)
    L0 = layers[0]
    q_h = L0.q.cpu().pin_memory()
    k_h = L0.ring_k[L0.slot:L0.slot + 1].cpu().pin_memory()
    v_h = L0.ring_v[L0.slot:L0.slot + 1].cpu().pin_memory()
    qi_h = L0.q_idx.cpu().pin_memory()
    out_h = torch.empty_like(L0.out, device="cpu").pin_memory()
    ins = [(q_h, lambda L: L.q), (k_h, lambda L: L.ring_k[L.slot:L.slot + 1]),
           (v_h, lambda L: L.ring_v[L.slot:L.slot + 1]), (qi_h, lambda L: L.q_idx)]
    h2d = sum(h.numel() * h.element_size() for h, _ in ins)
    d2h = out_h.numel() * out_h.element_size()
    rt = loaded_cudart()
    sh = stream.cuda_stream
    with torch.cuda.stream(stream):
        bound = [L.bind() for L in layers]
    copies = [[(dst(L).data_ptr(), h.data_ptr(), h.numel() * h.element_size()) for h, dst in ins] for L in layers]

    def one(t):
        L = layers[t % R]
        if rt is None:
            for h, dst in ins:
                dst(L).copy_(h, non_blocking=True)
            bound[t % R]()
            out_h.copy_(L.out, non_blocking=True)
            torch.cuda.current_stream().synchronize()
            return
        for dst, src, n in copies[t % R]:
            if rt.cudaMemcpyAsync(dst, src, n, 1, sh) != 0:
                raise RuntimeError("cudaMemcpyAsync (host to device) failed")
        bound[t % R]()
        if rt.cudaMemcpyAsync(out_h.data_ptr(), L.out.data_ptr(), d2h, 2, sh) != 0:
            raise RuntimeError("cudaMemcpyAsync (device to host) failed")
        if rt.cudaStreamSynchronize(sh) != 0:
            raise RuntimeError("cudaStreamSynchronize failed")

    with torch.cuda.stream(stream):
        for t in range(20):
            one(t)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for t in range(n_steps):
            one(t)
        dt = time.perf_counter() - t0
    assert ds4a.ds4a_last_device_error() == 0
    how = ("C-ABI calls marshalled once per layer (DecodeLayer.bind); "
           + ("cudaMemcpyAsync" if rt is not None else "torch copies")
           + " of q, new k/v and indexer query from pinned memory; D2H of out; stream sync each step; host clock")
    return {"value": round(n_steps / dt, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n_steps, "how": how}


def sub_decode(params, l2, stream, hbm_peak):
    import torch

    from compressed_sparse_mqa_gb300 import configs, timing
    from compressed_sparse_mqa_gb300.layer import DecodeLayer
    base = DecodeLayer(configs.decode(params))
    b = base.bytes_touched()
    R = rotation_copies(b, l2, minimum=8)
    layers = [base] + [base.clone() for _ in range(R - 1)]
    with torch.cuda.stream(stream):
        for L in layers[:2]:
            L.step()
    torch.cuda.synchronize()
    G = 1024
    g = timing.capture_graph(lambda t: layers[t % R].step(), G, stream)
    g.replay()
    ms = timing.time_graph(g, 8, stream)
    s = ms / 1e3 / (8 * G)
    return {"tokens_per_s_per_layer": round(1 / s, 1), "us_per_step": round(s * 1e6, 3),
            "bytes_per_step": b, "hbm_gbs": round(b / s / 1e9, 1), "hbm_frac": round(b / s / 1e9 / hbm_peak, 4),
            "rotation_copies": R}


def sub_prefill(params, l2, stream, peaks):
    import torch

    from compressed_sparse_mqa_gb300 import configs, timing
    from compressed_sparse_mqa_gb300.layer import PrefillLayer
    inst = configs.prefill(params)
    copies = [PrefillLayer(inst) for _ in range(3)]
    with torch.cuda.stream(stream):
        for L in copies:
            L.step()
    torch.cuda.synchronize()
    g = timing.capture_graph(lambda t: copies[t % 3].step(), 3, stream)
    g.replay()
    reps = 4
    ms = timing.time_graph(g, reps, stream)
    s = ms / 1e3 / (3 * reps)
    tflops = C4_FLOPS / s / 1e12
    peak = float(peaks.get("bf16_tflops", 1900.0))
    return {"tokens_per_s": round(inst.T / s, 1), "ms_per_chunk": round(s * 1e3, 4),
            "tflops": round(tflops, 2), "tensor_frac": round(tflops / peak, 4),
            "peak": f"{peak} TFLOP/s dense bf16 burst (fp16 runs at the same rate)",
            "flops_per_chunk": C4_FLOPS}


def sub_stack(l2, stream, hbm_peak):
    import torch

    from compressed_sparse_mqa_gb300 import configs, timing
    from compressed_sparse_mqa_gb300.layer import DecodeLayer
    stack = [DecodeLayer(configs.decode(configs.c5_layer_params(l))) for l in range(configs.C5_LAYERS)]
    b = sum(L.bytes_touched() for L in stack)
    n_copies = rotation_copies(b, l2, minimum=2)
    stacks = [stack] + [[L.clone() for L in stack] for _ in range(n_copies - 1)]
    with torch.cuda.stream(stream):
        for L in stack:
            L.step()
    torch.cuda.synchronize()

    def token(t):
        for L in stacks[t % n_copies]:
            L.step()

    G = 16
    g = timing.capture_graph(token, G, stream)
    g.replay()
    ms = timing.time_graph(g, 8, stream)
    s = ms / 1e3 / (8 * G)
    return {"us_per_token_43_layers": round(s * 1e6, 2), "tokens_per_s": round(1 / s, 1),
            "us_per_layer": round(s * 1e6 / configs.C5_LAYERS, 3), "bytes_per_token": b,
            "hbm_gbs": round(b / s / 1e9, 1), "hbm_frac": round(b / s / 1e9 / hbm_peak, 4),
            "rotation_copies": n_copies}


# ---------------------------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------------------------

def time_oracle_steps(inst, seconds: float, max_steps: int):
    import oracle
    oracle.decode_step(inst)   # build / warm
    n, t0 = 0, time.perf_counter()
    while n < max_steps and (time.perf_counter() - t0) < seconds:
        oracle.decode_step(inst)
        n += 1
    return n, time.perf_counter() - t0


def cpu_baseline(inst, seconds):
    n, dt = time_oracle_steps(inst, seconds, 10 ** 9)
    return {"value": round(n / dt, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} full C2 decode steps of the fp64 C oracle (single thread) in {dt:.1f} s"}


def run_reference(args, rank, world):
    from compressed_sparse_mqa_gb300 import configs
    if rank != 0:
        return None
    inst = configs.decode(configs.C2)
    budget = 120.0
    import oracle
    t0 = time.perf_counter()
    oracle.decode_step(inst)
    one = time.perf_counter() - t0
    warm = min(args.warmup, max(0, int(10.0 / max(one, 1e-6))))
    for _ in range(warm):
        oracle.decode_step(inst)
    n_max = max(1, min(args.steps, int(budget / max(one, 1e-6))))
    n, dt = time_oracle_steps(inst, budget, n_max)
    value = n / dt
    sample = f"{n} of {args.steps} requested full C2 decode steps (fp64 C oracle, 1 thread), {warm} warm-up"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": n, "warmup": warm, "ms_per_step": round(dt / n * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "C2 batch-1 decode, ratio-4 layer + indexer top-512, ctx 32768"},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "kind": "oracle", "cores": 1,
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
