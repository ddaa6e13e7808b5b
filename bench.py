#!/usr/bin/env python3
"""Benchmark of the compressed sparse MQA attention path on one GB300.

Headline step: one batch-1 decode token through one ratio-4 layer with the
indexer at context 32768 (8192 compressed rows, top-512, 128-row raw window, 64
heads, head_dim 128, fp16): ds4a_indexer_topk_compress (the indexer query and
the compressor's update for the new token, in one launch) -> ds4a_attn_decode.
Metric: tokens/s/layer (= steps/s) and the HBM bandwidth the step's algorithmic
bytes imply.

Inputs are resident in HBM.  The K timed steps (--steps) are one CUDA graph that
rotates over independent copies of the layer state (each step a different copy
while K is at most the number of copies).  Before every timed replay of that
graph a write of twice the L2 size evicts the L2, so every step streams its keys
and rows from DRAM; the replay is timed with CUDA events on its stream, and the
measurement is repeated (--samples) to report the median and its spread.

Printed (one JSON line on rank 0): the headline metric, e2e (the same step
through the C ABI with the step's inputs copied from pinned host memory and the
output read back, every step), the roofline of the dominant kernel, the oracle's
CPU time on the host's cores, the clocks seen, and sub-results for the ratio-128
decode layer, the 2048-token prefill chunk and the 43-layer decode stack.
`--impl reference` times the fp64 CPU oracle on the same step instead.
"""
from __future__ import annotations

import argparse
import ctypes
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
    ap.add_argument("--steps", type=int, default=256, help="steps per timed region (one CUDA graph)")
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--samples", type=int, default=100,
                    help="timed regions (each after an L2 flush); the median is reported")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sub", action="store_true", help="skip the C3/C4/C5 sub-results")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", choices=["c3", "c4", "c5", "prefill_stack", "batched16", "batched64"], default=None,
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

def timed_graph(fn, steps, stream):
    """A CUDA graph of fn(0) .. fn(G-1) with G the largest divisor of `steps` up to 1024,
    and the number of back-to-back replays that make `steps` steps."""
    from compressed_sparse_mqa_gb300 import timing
    G = graph_size(steps)
    g = timing.capture_graph(fn, G, stream)
    return g, steps // G


def sampled(g, replays, steps, samples, stream, flush):
    """Per-step milliseconds of each timed region: an L2 flush, then `replays`
    replays of g (= `steps` steps), events on `stream`."""
    from compressed_sparse_mqa_gb300 import timing
    g.replay()   # upload and warm
    ms = timing.time_graph_samples(g, samples, stream, flush, replays)
    return [m / steps for m in ms]


def run_ours(args, rank, world, local):
    import torch

    from compressed_sparse_mqa_gb300 import configs, ds4a, timing
    from compressed_sparse_mqa_gb300.layer import DecodeLayer

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
    flush = timing.L2Flush()
    if args.only:
        fn = {"c3": lambda: sub_decode(configs.C3, l2, stream, hbm_peak, flush),
              "c4": lambda: sub_prefill(configs.C4, stream, peaks, flush),
              "c5": lambda: sub_stack(l2, stream, hbm_peak, flush),
              "prefill_stack": lambda: sub_prefill_stack(stream, peaks, flush),
              "batched16": lambda: sub_batched(16, l2, stream, hbm_peak, flush),
              "batched64": lambda: sub_batched(64, l2, stream, hbm_peak, flush)}[args.only]
        return {"only": args.only, "result": fn()}

    # ---- headline: C2 decode step --------------------------------------------------------
    inst = configs.decode(configs.C2)
    base = DecodeLayer(inst)
    step_bytes = base.bytes_touched()
    R = rotation_copies(step_bytes, l2, minimum=8)
    layers = [base] + [base.clone() for _ in range(R - 1)]
    K, W = max(1, args.steps), max(3, args.warmup)
    with torch.cuda.stream(stream):
        for t in range(W):          # warm-up steps, untimed
            layers[t % R].step()
    torch.cuda.synchronize()
    g, reps = timed_graph(lambda t: layers[t % R].step(), K, stream)
    n_samples = max(1, args.samples)
    barrier(world)
    with timing.ClockSampler(local) as clk:
        per_step = sampled(g, reps, K, n_samples, stream, flush)
    barrier(world)
    clocks = clk.summary()
    sp = timing.spread(per_step)
    ms_step, value = job_throughput(sp["median"], 1, world)
    s_per_step = ms_step / 1e3
    gbs = step_bytes / s_per_step / 1e9

    # ---- per-kernel durations (each kernel alone, events on the launching stream) --------
    def k_prep(t):
        L = layers[t % R]
        ds4a.ds4a_indexer_topk_compress(L.q_idx, L.kidx, L.p, L.ratio, L.topk, L.sel, L.sel_n, L.ws,
                                        L.ring_k[L.slot:L.slot + 1], L.ring_v[L.slot:L.slot + 1], L.w, L.state,
                                        L.comp_k, L.comp_v)

    def k_attn(t):
        L = layers[t % R]
        ds4a.ds4a_attn_decode(L.q, L.ring_k[:L.n_win], L.ring_v[:L.n_win], L.comp_k, L.comp_v, L.sel, L.topk,
                              L.scale, L.out)

    # a graph of n_k back-to-back launches of one kernel over the rotation, timed after an
    # L2 flush; average per launch, median over samples
    n_k = min(K, R)
    kt = {}
    for name, fn in [("indexer_topk_compress", k_prep), ("attn_decode", k_attn)]:
        gk, rk = timed_graph(fn, n_k, stream)
        kt[name] = timing.spread(sampled(gk, rk, n_k, 20, stream, flush))["median"]
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
                "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
                "kernel_us": {k: round(v * 1e3, 3) for k, v in kt.items()},
                "kernel_bytes": kbytes,
                "how": f"each kernel alone: graph of {n_k} launches over the layer copies after an L2 flush, "
                       f"median of 20 samples per launch"}

    # ---- e2e: per-step inputs from pinned host memory, output read back every step ----------
    e2e = run_e2e(layers, stream, n_steps=max(200, min(2000, K * 4)))

    # ---- sub-results ---------------------------------------------------------------------------
    sub = {}
    if not args.no_sub:
        sub["c3_decode_ratio128_ctx131072"] = sub_decode(configs.C3, l2, stream, hbm_peak, flush)
        sub["c2_pooled_indexer_keys"] = sub_decode(configs.C2_POOLED, l2, stream, hbm_peak, flush)
        sub["batched_decode_16_sessions_c2"] = sub_batched(16, l2, stream, hbm_peak, flush)
        sub["batched_decode_64_sessions_c2"] = sub_batched(64, l2, stream, hbm_peak, flush)
        sub["c4_prefill_2048_ratio4"] = sub_prefill(configs.C4, stream, peaks, flush)
        sub["c5_stack_43_layers_ctx65536"] = sub_stack(l2, stream, hbm_peak, flush)
        sub["prefill_stack_43_layers_2048_after_30720"] = sub_prefill_stack(stream, peaks, flush)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 (fp32 accumulate)",
        "data": "synthetic (seeded SplitMix64/Box-Muller, N(0,1) values)",
        "config": {"workload": "C2 batch-1 decode, ratio-4 layer + indexer top-512, ctx 32768",
                   "heads": H, "kv_heads": 1, "head_dim": D, "window": base.W, "compressed_rows": base.n_vis,
                   "topk": base.topk, "index_dim": base.kidx.shape[1],
                   "l2_policy": f"L2 flushed (write of {flush.nbytes / 1e6:.0f} MB = 2x L2) before every timed "
                                f"region; the {K} steps of a region rotate over {R} layer copies "
                                f"({R * step_bytes / 1e6:.0f} MB), "
                                + ("so no step's data is in L2 from an earlier step" if K <= R else
                                   "each copy reused after the other copies evicted it"),
                   "timed_region": f"CUDA graph of {K // reps} steps x {reps} replay(s) = {K} steps, CUDA events "
                                   f"on its stream; {n_samples} regions, median reported",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "spread_us_per_step": {k: (round(v * 1e3, 3) if k != "n" else v) for k, v in sp.items()},
        "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4), "bytes_per_step": step_bytes,
        "e2e": e2e, "gpu_launches": launches_per_step * K * n_samples, "roofline": roofline, "clocks": clocks,
        "sub": sub,
    }
    if rank == 0 and args.cpu_seconds > 0:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


def run_e2e(layers, stream, n_steps):
    """Steps through the public API with the step's inputs in pinned host memory and the
    output read back, every step, on the host clock: one ds4a_decode_layer_step call per
    step copies the token's K and V, the query and the indexer query in, runs the
    layer's launches, copies the output out and waits for it (DecodeLayer.bind_host
    marshals each layer copy's call once)."""
    import torch

    from compressed_sparse_mqa_gb300 import ds4a
    R = len(layers)
    L0 = layers[0]
    # the step's inputs live in one page-locked block (q, k, v, the indexer query and,
    # with pooled keys, the token's indexer key), each a view at a 16-byte offset
    parts = [L0.q, L0.ring_k[L0.slot], L0.ring_v[L0.slot]] + ([L0.q_idx] if L0.topk else []) + \
        ([L0.ki_tok] if L0.pooled_keys else [])
    sizes = [t.numel() for t in parts]
    offs = [sum((n + 7) // 8 * 8 for n in sizes[:i]) for i in range(len(sizes))]
    block = torch.empty(offs[-1] + (sizes[-1] + 7) // 8 * 8, dtype=torch.float16).pin_memory()
    views = [block[o:o + n] for o, n in zip(offs, sizes)]
    for v, t in zip(views, parts):
        v.copy_(t.reshape(-1).cpu())
    q_h, k_h, v_h = views[0], views[1], views[2]
    qi_h = views[3] if L0.topk else None
    kt_h = views[-1] if L0.pooled_keys else None
    out_h = torch.empty_like(L0.out, device="cpu").pin_memory()
    h2d = sum(n * 2 for n in sizes)
    d2h = out_h.numel() * out_h.element_size()
    bound = [L.bind_host(k_h, v_h, q_h, qi_h, out_h, ki_tok=kt_h, stream=stream) for L in layers]
    # each step's inputs are written into the pinned block by the host first, as a
    # caller producing them would (so no step reads inputs the GPU has seen before)
    src = block.clone()
    dst_p, src_p, nbytes = block.data_ptr(), src.data_ptr(), block.numel() * 2

    def one(t):
        ctypes.memmove(dst_p, src_p, nbytes)
        bound[t % R]()

    with torch.cuda.stream(stream):
        for t in range(20):
            one(t)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for t in range(n_steps):
            one(t)
        dt = time.perf_counter() - t0
    assert ds4a.ds4a_last_device_error() == 0
    how = ("per step: the host writes the token's K and V, q and the indexer query into one pinned block, then one "
           "ds4a_decode_layer_step call (marshalled once per layer copy): a kernel reads the pinned inputs over "
           "the host link into the layer's arrays, the step's launches, the attention kernel writes out into a "
           "pinned buffer, stream sync; host clock")
    return {"value": round(n_steps / dt, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n_steps, "how": how}


def sub_decode(params, l2, stream, hbm_peak, flush):
    import torch

    from compressed_sparse_mqa_gb300 import configs, timing
    from compressed_sparse_mqa_gb300.layer import DecodeLayer
    base = DecodeLayer(configs.decode(params))
    b = base.bytes_touched()
    R = rotation_copies(b, l2, minimum=8)
    layers = [base] + [base.clone() for _ in range(R - 1)]
    with torch.cuda.stream(stream):
        for L in layers[:4]:
            L.step()
    torch.cuda.synchronize()
    K = min(256, R)
    g, reps = timed_graph(lambda t: layers[t % R].step(), K, stream)
    sp = timing.spread(sampled(g, reps, K, 30, stream, flush))
    s = sp["median"] / 1e3
    return {"tokens_per_s_per_layer": round(1 / s, 1), "us_per_step": round(s * 1e6, 3),
            "us_p10_p90": [round(sp["p10"] * 1e3, 3), round(sp["p90"] * 1e3, 3)],
            "bytes_per_step": b, "hbm_gbs": round(b / s / 1e9, 1), "hbm_frac": round(b / s / 1e9 / hbm_peak, 4),
            "timed": f"graph of {K} steps over {R} layer copies, L2 flushed before each of 30 regions, median"}


def sub_prefill(params, stream, peaks, flush):
    import torch

    from compressed_sparse_mqa_gb300 import configs, timing
    from compressed_sparse_mqa_gb300.layer import PrefillLayer
    inst = configs.prefill(params)
    copies = [PrefillLayer(inst) for _ in range(2)]
    with torch.cuda.stream(stream):
        for L in copies:
            L.step()
    torch.cuda.synchronize()
    g, reps = timed_graph(lambda t: copies[t % 2].step(), 2, stream)
    sp = timing.spread(sampled(g, reps, 2, 10, stream, flush))
    s = sp["median"] / 1e3
    tflops = C4_FLOPS / s / 1e12
    peak = float(peaks.get("bf16_tflops", 1900.0))
    return {"tokens_per_s": round(inst.T / s, 1), "ms_per_chunk": round(s * 1e3, 4),
            "tflops": round(tflops, 2), "tensor_frac": round(tflops / peak, 4),
            "peak": f"{peak} TFLOP/s dense bf16 burst, measured (fp16 runs at the same rate)",
            "flops_per_chunk": C4_FLOPS,
            "timed": "graph of 2 chunks (2 copies), L2 flushed before each of 10 regions, median",
            "attention_gather": prefill_gather_roofline(copies, stream, flush)}


def prefill_gather_roofline(copies, stream, flush):
    """The prefill attention kernel against the rate at which rows can be gathered: every
    query reads its window rows and its kept compressed rows (K and V, 256 B each).  The
    peak is measured here with ds4a_probe_gather (16-byte asynchronous copies of rows
    by index into shared memory, nothing else) on the chunk's own kept-row lists over
    its compressed K rows, after an L2 flush, median of 10."""
    import torch

    from compressed_sparse_mqa_gb300 import ds4a, timing
    L = copies[0]
    T, D = L.T, L.D
    n_win = sum(min(L.W, L.P + i + 1) for i in range(T))
    n_sel = int((L.sel >= 0).sum().item())
    row = D * 2
    gathered = 2 * (n_win + n_sel) * row            # K and V rows read by the kernel

    def attn(t):
        C = copies[t % 2]
        ds4a.ds4a_attn_prefill(C.q, C.raw_k, C.raw_v, C.n_prior, C.W, C.comp_k, C.comp_v, C.sel, C.P, C.ratio,
                               C.scale, C.out)

    g, reps = timed_graph(attn, 2, stream)
    t_attn = timing.spread(sampled(g, reps, 2, 10, stream, flush))["median"] / 1e3
    idx = L.sel.clamp(min=0).reshape(-1).contiguous()
    sink = torch.zeros(1, dtype=torch.int32, device=idx.device)
    gp, rp = timed_graph(lambda t: ds4a.ds4a_probe_gather(L.comp_k, idx, sink), 2, stream)
    t_probe = timing.spread(sampled(gp, rp, 2, 10, stream, flush))["median"] / 1e3
    peak = idx.numel() * row / t_probe
    achieved = gathered / t_attn
    return {"bytes_gathered": gathered, "attention_us": round(t_attn * 1e6, 2),
            "achieved_tbs": round(achieved / 1e12, 3), "gather_peak_tbs": round(peak / 1e12, 3),
            "frac": round(achieved / peak, 4), "probe_us": round(t_probe * 1e6, 2),
            "peak_how": "ds4a_probe_gather: the chunk's 1,048,576 kept-row indices over its compressed K rows, "
                        "16-byte cp.async into shared memory, L2 flushed first, median of 10"}


def sub_batched(B, l2, stream, hbm_peak, flush):
    """B independent C2-shaped sessions (ratio-4 layer + indexer, context 32768, each
    session its own seeded cache) decoded together: one batched indexer launch and one
    batched attention launch per step."""
    import torch

    from compressed_sparse_mqa_gb300 import configs, timing
    from compressed_sparse_mqa_gb300.layer import BatchedDecodeLayer
    import dataclasses
    insts = [configs.decode(dict(configs.C2, seed=s)) for s in range(B)]
    insts = [dataclasses.replace(i, w=insts[0].w) for i in insts]   # one layer: shared score weights
    base = BatchedDecodeLayer(insts)
    b = base.bytes_touched()
    R = rotation_copies(b, l2, minimum=2)
    layers = [base] + [base.clone() for _ in range(R - 1)]
    with torch.cuda.stream(stream):
        for L in layers:
            L.step()
    torch.cuda.synchronize()
    K = R
    g, reps = timed_graph(lambda t: layers[t % R].step(), K, stream)
    sp = timing.spread(sampled(g, reps, K, 30, stream, flush))
    s = sp["median"] / 1e3
    # each of the step's two launches alone, over the copies, after an L2 flush
    from compressed_sparse_mqa_gb300 import ds4a
    kernel_us = {}
    for name in ("ds4a_indexer_topk_compress_batched", "ds4a_attn_decode_batched"):
        calls = [dict(L._step_calls())[name] for L in layers]
        gk, rk = timed_graph(lambda t: getattr(ds4a, name)(*calls[t % R]), K, stream)
        kernel_us[name] = round(timing.spread(sampled(gk, rk, K, 20, stream, flush))["median"] * 1e3, 3)
    return {"sessions": B, "tokens_per_s": round(B / s, 1), "us_per_step": round(s * 1e6, 3),
            "us_per_token_layer": round(s * 1e6 / B, 3), "bytes_per_step": b,
            "hbm_gbs": round(b / s / 1e9, 1), "hbm_frac": round(b / s / 1e9 / hbm_peak, 4),
            "kernel_us": kernel_us,
            "timed": f"graph of {K} batched steps over {R} copies, L2 flushed before each of 30 regions, median"}


def sub_prefill_stack(stream, peaks, flush):
    """One 2048-token chunk through all 43 layers (window only, ratio 4 + indexer,
    ratio 128), every layer's state resident; the flops are the algorithmic flops of
    every layer's indexer GEMM and attention."""
    import torch

    from compressed_sparse_mqa_gb300 import configs, timing
    from compressed_sparse_mqa_gb300.layer import PrefillStack
    insts = configs.prefill_stack()
    flops = sum(configs.prefill_flops(i) for i in insts)
    stack = PrefillStack(insts)
    with torch.cuda.stream(stream):
        stack.step()
    torch.cuda.synchronize()
    g, reps = timed_graph(lambda t: stack.step(), 1, stream)
    sp = timing.spread(sampled(g, reps, 1, 8, stream, flush))
    s = sp["median"] / 1e3
    tflops = flops / s / 1e12
    sus = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0)))
    return {"tokens_per_s": round(insts[0].T / s, 1), "ms_per_chunk_43_layers": round(s * 1e3, 3),
            "tflops": round(tflops, 2), "tensor_frac_sustained": round(tflops / sus, 4),
            "peak": f"{sus} TFLOP/s dense bf16 sustained, measured (fp16 runs at the same rate)",
            "flops_per_chunk": flops, "prefix_tokens": insts[0].P, "chunk_tokens": insts[0].T,
            "timed": "graph of one chunk through 43 layers, L2 flushed before each of 8 regions, median"}


def sub_stack(l2, stream, hbm_peak, flush):
    import torch

    from compressed_sparse_mqa_gb300 import configs, timing
    from compressed_sparse_mqa_gb300.layer import DecodeLayer
    stack = [DecodeLayer(configs.decode(configs.c5_layer_params(l))) for l in range(configs.C5_LAYERS)]
    b = sum(L.bytes_touched() for L in stack)
    n_copies = 2
    stacks = [stack] + [[L.clone() for L in stack] for _ in range(n_copies - 1)]
    with torch.cuda.stream(stream):
        for L in stack:
            L.step()
    torch.cuda.synchronize()

    def token(t):
        for L in stacks[t % n_copies]:
            L.step()

    g, reps = timed_graph(token, 2, stream)
    sp = timing.spread(sampled(g, reps, 2, 20, stream, flush))
    s = sp["median"] / 1e3
    return {"us_per_token_43_layers": round(s * 1e6, 2), "tokens_per_s": round(1 / s, 1),
            "us_per_layer": round(s * 1e6 / configs.C5_LAYERS, 3), "bytes_per_token": b,
            "hbm_gbs": round(b / s / 1e9, 1), "hbm_frac": round(b / s / 1e9 / hbm_peak, 4),
            "timed": "graph of 2 tokens (2 copies of the stack, 206 MB), L2 flushed before each of 20 regions, median"}


# ---------------------------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------------------------

def cpu_info() -> dict:
    """Model name and maximum clock of the host's CPU, as far as the OS reports them."""
    info = {"model": None, "max_ghz": None}
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and info["model"] is None:
                info["model"] = v.strip()
            if k.strip() == "CPU max MHz":
                info["max_ghz"] = round(float(v.strip()) / 1e3, 3)
    except (OSError, ValueError):
        pass
    if info["max_ghz"] is None:
        try:
            with open("/sys/devices/system/cpu/cpu0/cpufreq/cpuinfo_max_freq") as f:
                info["max_ghz"] = round(int(f.read()) / 1e6, 3)
        except (OSError, ValueError):
            pass
    return info


def _oracle_worker(args):
    """One process: build the C2 step's inputs, wait for the others, then run full
    oracle decode steps until `seconds` pass or `max_steps` are done."""
    seconds, max_steps, barrier_ = args
    sys.path.insert(0, ROOT)
    import oracle
    from compressed_sparse_mqa_gb300 import configs
    inst = configs.decode(configs.C2)
    oracle.decode_step(inst)   # warm
    barrier_.wait()
    n, t0 = 0, time.perf_counter()
    while n < max_steps and (time.perf_counter() - t0) < seconds:
        oracle.decode_step(inst)
        n += 1
    return n, time.perf_counter() - t0


def oracle_steps_all_cores(seconds: float, max_steps_total: int):
    """Full C2 oracle steps run by one process per usable core (spawned, so that no
    CUDA state is inherited); returns (steps, seconds, processes)."""
    import multiprocessing as mp
    n = cpu_cores()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        bar = m.Barrier(n)
        per = max(1, math.ceil(max_steps_total / n))
        with ctx.Pool(n) as pool:
            res = pool.map(_oracle_worker, [(seconds, per, bar)] * n)
    steps = sum(r[0] for r in res)
    return steps, max(r[1] for r in res), n


def time_oracle_steps(inst, seconds: float, max_steps: int):
    import oracle
    oracle.decode_step(inst)   # build / warm
    n, t0 = 0, time.perf_counter()
    while n < max_steps and (time.perf_counter() - t0) < seconds:
        oracle.decode_step(inst)
        n += 1
    return n, time.perf_counter() - t0


def oracle_prefill_sample(n_q: int = 64):
    """The oracle on the first n_q queries of the 2048-token prefill chunk (the same
    inputs, the chunk cut after n_q queries): tokens/s on one core."""
    import dataclasses

    import oracle
    from compressed_sparse_mqa_gb300 import configs
    inst = configs.prefill(configs.C4)
    r = inst.ratio
    sub = dataclasses.replace(inst, T=n_q, raw_k=inst.raw_k[: inst.n_prior + n_q],
                              raw_v=inst.raw_v[: inst.n_prior + n_q], kidx=inst.kidx[: (inst.P + n_q) // r],
                              q=inst.q[:n_q], q_idx=inst.q_idx[:n_q])
    t0 = time.perf_counter()
    oracle.prefill_chunk(sub)
    dt = time.perf_counter() - t0
    return {"tokens_per_s": round(n_q / dt, 2), "cores": 1,
            "sample": f"first {n_q} of the 2048 queries of the prefill chunk (compressor, indexer, attention), "
                      f"fp64 C oracle, one thread, {dt:.1f} s"}


def cpu_baseline(seconds):
    """The oracle as it stands on the host: full C2 steps on one core and on every
    usable core (one process each), and a bounded sample of the prefill chunk."""
    import oracle
    from compressed_sparse_mqa_gb300 import configs
    inst = configs.decode(configs.C2)
    n1, dt1 = time_oracle_steps(inst, seconds, 10 ** 9)
    nn, dtn, procs = oracle_steps_all_cores(seconds, 10 ** 9)
    info = cpu_info()
    return {"value": round(nn / dtn, 3), "unit": UNIT, "cores": procs, "kind": "oracle",
            "sample": f"{nn} full C2 decode steps of the fp64 C oracle in {dtn:.1f} s, one process per usable "
                      f"core ({procs})",
            "single_thread": {"value": round(n1 / dt1, 3), "unit": UNIT,
                              "sample": f"{n1} full C2 steps in {dt1:.1f} s on one core"},
            "cpu": info, "c4_prefill": oracle_prefill_sample()}


def _oracle_round_worker(args):
    """One process: `warmup` untimed full C2 oracle steps (at least one, which builds the
    inputs), then, once every process is ready, `steps` timed ones; returns their seconds."""
    warmup, steps, barrier_ = args
    sys.path.insert(0, ROOT)
    import oracle
    from compressed_sparse_mqa_gb300 import configs
    inst = configs.decode(configs.C2)
    for _ in range(max(1, warmup)):
        oracle.decode_step(inst)
    barrier_.wait()
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.decode_step(inst)
    return time.perf_counter() - t0


def oracle_rounds_all_cores(steps: int, warmup: int):
    """`steps` timed rounds after `warmup` untimed ones, a round being one full C2 oracle
    step on each usable core (one spawned process per core); returns (seconds, processes)."""
    import multiprocessing as mp
    n = cpu_cores()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        bar = m.Barrier(n)
        with ctx.Pool(n) as pool:
            res = pool.map(_oracle_round_worker, [(warmup, steps, bar)] * n)
    return max(res), n


def run_reference(args, rank, world):
    if rank != 0:
        return None
    K, W = max(1, args.steps), max(0, args.warmup)
    dtn, procs = oracle_rounds_all_cores(K, W)
    nn = K * procs   # tokens: one C2 step per core per round
    value = nn / dtn
    sample = (f"{K} timed rounds after {W} untimed ones (each process builds its inputs with at least one); a "
              f"round is one full C2 decode step of the fp64 C oracle on each of the {procs} usable cores (one "
              f"process per core), so {nn} steps in {dtn:.2f} s")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(dtn / K * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "C2 batch-1 decode, ratio-4 layer + indexer top-512, ctx 32768"},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "kind": "oracle", "cores": procs,
                             "sample": sample, "cpu": cpu_info()},
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
