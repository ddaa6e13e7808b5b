"""The five workloads, shaped like the DeepSeek-V4-Flash attention layers the
"DS4 (DwarfStar 4)" page describes (Architecture: 43 layers, 64 heads, 1 KV head,
128-token window, 4096-dim model; prefill chunks of 2048 tokens).

All inputs are seeded synthetic draws (compressed_sparse_mqa_gb300.synth):
values N(0, 1), compressor score weights N(0, 1/128) on the full-size layers.
"""
from __future__ import annotations

import math

from . import synth
from .layer import layer_schedule

SIGMA_W = math.sqrt(1.0 / 128.0)

# tiny even-layer instance: the oracle finishes it in well under a second
C1 = dict(seed=0, layer=0, H=8, D=64, window=32, ratio=4, d_idx=32, topk=16, p=512,
          pooled_history=True, sigma_w=1.0)
# batch-1 decode, ratio-4 layer with indexer, context 32768 (8192 compressed rows)
C2 = dict(seed=0, layer=0, H=64, D=128, window=128, ratio=4, d_idx=128, topk=512, p=32768,
          sigma_w=SIGMA_W)
# the same step when the compressor pools per-token indexer keys into the rows' keys
C2_POOLED = dict(C2, pooled_keys=True)
# batch-1 decode, ratio-128 layer, context 131072 (1024 compressed rows, all attended)
C3 = dict(seed=0, layer=0, H=64, D=128, window=128, ratio=128, d_idx=128, topk=0, p=131072,
          sigma_w=SIGMA_W)
# the same layer one token earlier: this step completes block 1023 and appends its row
C3_EMIT = dict(C3, p=131071)
# prefill chunk: 2048 tokens after a 30720-token prefix on a ratio-4 layer
C4 = dict(seed=0, layer=0, H=64, D=128, window=128, ratio=4, d_idx=128, topk=512, P=30720, T=2048,
          sigma_w=SIGMA_W)
# full 43-layer decode stack at context 65536
C5_CONTEXT = 65536
C5_LAYERS = 43


def c5_layer_params(layer: int, context: int = C5_CONTEXT) -> dict:
    ratio, topk = layer_schedule(layer)
    return dict(seed=layer, layer=layer, H=64, D=128, window=128, ratio=ratio, d_idx=128, topk=topk,
                p=context, sigma_w=SIGMA_W)


# 43-layer prefill of one 2048-token chunk after a 30720-token prefix: every layer
# with its schedule (window only, ratio 4 + top-512, ratio 128); the chunk's queries
# are one draw fed to every layer, each layer's cache, indexer keys and score
# weights are its own draw (seed = layer)
PREFILL_STACK_P = 30720
PREFILL_STACK_T = 2048


def prefill_stack_layer_params(layer: int, P: int = PREFILL_STACK_P, T: int = PREFILL_STACK_T) -> dict:
    ratio, topk = layer_schedule(layer)
    return dict(seed=layer, layer=layer, H=64, D=128, window=128, ratio=ratio, d_idx=128, topk=topk, P=P, T=T,
                sigma_w=SIGMA_W)


def prefill_stack(P: int = PREFILL_STACK_P, T: int = PREFILL_STACK_T, layers=None) -> list:
    """PrefillInstances of the stack's layers (all 43 unless `layers` lists some)."""
    queries = synth.chunk_queries(0, T, 64, 128, 128)
    ids = range(C5_LAYERS) if layers is None else layers
    return [synth.prefill_instance(**prefill_stack_layer_params(l, P, T), queries=queries) for l in ids]


def prefill_flops(inst) -> float:
    """Algorithmic flops of one prefill chunk of one layer: the causal indexer GEMM
    (2 d_idx per visible row and query) and attention (4 D per head, query and
    attended row: QK^T and PV), each query attending its window rows and its kept
    (or every visible) compressed row."""
    f = 0.0
    for i in range(inst.T):
        p = inst.P + i
        n_win = min(inst.window, p + 1)
        n_vis = (p + 1) // inst.ratio if inst.ratio else 0
        if inst.topk:
            f += 2.0 * inst.d_idx * n_vis
        n_comp = min(inst.topk, n_vis) if inst.topk else n_vis
        f += 4.0 * inst.H * inst.D * (n_win + n_comp)
    return f


def decode(params: dict) -> synth.DecodeInstance:
    return synth.decode_instance(**params)


def prefill(params: dict) -> synth.PrefillInstance:
    return synth.prefill_instance(**params)
