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


def decode(params: dict) -> synth.DecodeInstance:
    return synth.decode_instance(**params)


def prefill(params: dict) -> synth.PrefillInstance:
    return synth.prefill_instance(**params)
