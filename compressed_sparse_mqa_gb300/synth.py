"""Seeded synthetic inputs for the compressed sparse MQA attention path.

This module only draws random numbers and lays them out in the shapes of the
DS4 / DeepSeek-V4-Flash attention layers ("DS4 (DwarfStar 4)" page, Architecture:
64 query heads, 1 KV head, 128-token sliding window, 4096-dim model; Key
Techniques, "KV attention compression": ratio 4 / 128 layers, top-512 indexer).
It holds none of the method's arithmetic, so both the CUDA path and the CPU
oracle can be fed from it without sharing any code of the method.

Generator (one independent stream per tensor):
  * SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): state += 0x9E3779B97F4A7C15, then the
    (30, 27, 31) xor-shift-multiply finaliser.
  * 53-bit uniforms: u = (z >> 11) * 2^-53.
  * Box-Muller (1958) in double on consecutive pairs (u1 taken in (0, 1]).
  * scale by sigma, round once to fp16 with round-to-nearest-even.
Stream seed: splitmix64_mix(seed ^ (layer << 32) ^ tensor_id) with the tensor
ids below.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15

# one stream per tensor kind
T_Q, T_KRAW, T_VRAW, T_COMPK, T_COMPV, T_KIDX, T_QIDX, T_W = 1, 2, 3, 4, 5, 6, 7, 8
# per-token indexer keys (the reading in which the compressor pools them into the rows' keys)
T_KIDX_TOK = 9


def _mix_scalar(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def _mix_array(z: np.ndarray) -> np.ndarray:
    # numpy uint64 array arithmetic wraps modulo 2^64
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def stream_seed(seed: int, layer: int, tensor_id: int) -> int:
    return _mix_scalar((seed ^ (layer << 32) ^ tensor_id) & MASK64)


def raw_u64(stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset .. offset+n-1 of the SplitMix64 stream starting at `stream`."""
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        states = np.uint64(stream) + i * np.uint64(GOLDEN)
    return _mix_array(states)


def uniforms(stream: int, n: int) -> np.ndarray:
    return (raw_u64(stream, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals(stream: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """n draws of N(0, sigma^2) in double (Box-Muller on consecutive pairs)."""
    m = (n + 1) // 2
    z = raw_u64(stream, 2 * m)
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n] * sigma


def normal_f16(seed: int, layer: int, tensor_id: int, shape, sigma: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    x = normals(stream_seed(seed, layer, tensor_id), n, sigma)
    return x.astype(np.float16).reshape(shape)   # numpy double->half is RNE


def normal_f32(seed: int, layer: int, tensor_id: int, shape, sigma: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    x = normals(stream_seed(seed, layer, tensor_id), n, sigma)
    return x.astype(np.float32).reshape(shape)


# ----------------------------------------------------------------------------
# Instances: one decode step of one layer, or one prefill chunk of one layer.
# Every parameter that shapes the draw (ratio, window, top-k) is passed in; the
# layer schedule itself lives with the code that runs the method.
# ----------------------------------------------------------------------------

@dataclass
class DecodeInstance:
    """Inputs of one batch-1 decode step for one layer at absolute position p.

    raw_k/raw_v  [n_raw, D] fp16: tokens at positions raw_pos0 .. p (the raw
                 window and the tokens of the compressor's open block).
    comp_k/comp_v [n_given, D] fp16: pooled rows that exist before this step
                 (given data), or empty when `pooled_history` is set, in which
                 case raw_k/raw_v hold every position 0 .. p and the rows come
                 from running the compressor over them.
    kidx [n_vis, d_i] fp16: one indexer key per compressed row visible to p; with
                 pooled keys, the keys of the given rows only.
    kidx_tok [n_raw, d_i] fp16 or None: with pooled keys, the indexer key of every
                 raw token (positions raw_pos0 .. p), which the compressor pools into
                 the keys of the rows they complete.
    q [H, D] fp16, q_idx [d_i] fp16, w [D] fp32 (compressor score weights).
    """
    H: int
    D: int
    window: int
    ratio: int
    d_idx: int
    topk: int
    p: int
    pooled_history: bool
    raw_pos0: int
    raw_k: np.ndarray
    raw_v: np.ndarray
    comp_k: np.ndarray
    comp_v: np.ndarray
    kidx: np.ndarray
    q: np.ndarray
    q_idx: np.ndarray
    w: np.ndarray
    kidx_tok: "np.ndarray | None" = None
    meta: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def decode_instance(*, seed: int, layer: int, H: int, D: int, window: int, ratio: int,
                    d_idx: int, topk: int, p: int, pooled_history: bool = False,
                    sigma_w: float = 1.0, pooled_keys: bool = False) -> DecodeInstance:
    """Draw the inputs of one decode step (all values N(0,1) except w ~ N(0, sigma_w^2)).

    ratio == 0 means a raw-window-only layer (no compressed rows, no indexer);
    topk == 0 means no indexer (every visible compressed row is attended);
    pooled_keys: the rows' indexer keys are pooled from per-token keys (drawn for
    every raw token), and only the given rows' keys are drawn directly.
    """
    if pooled_history:
        raw_pos0 = 0
    else:
        first_open = (p // ratio) * ratio if ratio > 0 else p
        raw_pos0 = max(0, min(p - window + 1, first_open))
    n_raw = p - raw_pos0 + 1
    n_given = 0 if (pooled_history or ratio == 0) else p // ratio
    n_vis = (p + 1) // ratio if ratio > 0 else 0
    raw_k = normal_f16(seed, layer, T_KRAW, (n_raw, D))
    raw_v = normal_f16(seed, layer, T_VRAW, (n_raw, D))
    comp_k = normal_f16(seed, layer, T_COMPK, (n_given, D))
    comp_v = normal_f16(seed, layer, T_COMPV, (n_given, D))
    n_keys = (n_given if pooled_keys else n_vis) if topk > 0 else 0
    kidx = normal_f16(seed, layer, T_KIDX, (n_keys, d_idx))
    kidx_tok = normal_f16(seed, layer, T_KIDX_TOK, (n_raw, d_idx)) if (pooled_keys and topk > 0) else None
    q = normal_f16(seed, layer, T_Q, (H, D))
    q_idx = normal_f16(seed, layer, T_QIDX, (d_idx if topk > 0 else 0,))
    w = normal_f32(seed, layer, T_W, (D,), sigma_w)
    return DecodeInstance(H=H, D=D, window=window, ratio=ratio, d_idx=d_idx, topk=topk,
                          p=p, pooled_history=pooled_history, raw_pos0=raw_pos0,
                          raw_k=raw_k, raw_v=raw_v, comp_k=comp_k, comp_v=comp_v,
                          kidx=kidx, q=q, q_idx=q_idx, w=w, kidx_tok=kidx_tok)


@dataclass
class PrefillInstance:
    """Inputs of one prefill chunk of T tokens appended after a prefix of P tokens.

    raw_k/raw_v [n_prior + T, D] fp16: the last n_prior prefix tokens (at least
                min(window-1, P), and every token of the prefix's open block), then
                the T chunk tokens (positions P - n_prior .. P+T-1).
    comp_k/comp_v [P // ratio, D] fp16: the prefix's pooled rows (given data).
    kidx [(P+T) // ratio, d_i] fp16: indexer keys of every row visible by the
                chunk's end (prefix rows and the rows the chunk completes).
    q [T, H, D] fp16, q_idx [T, d_i] fp16, w [D] fp32.
    """
    H: int
    D: int
    window: int
    ratio: int
    d_idx: int
    topk: int
    P: int
    T: int
    n_prior: int
    raw_k: np.ndarray
    raw_v: np.ndarray
    comp_k: np.ndarray
    comp_v: np.ndarray
    kidx: np.ndarray
    q: np.ndarray
    q_idx: np.ndarray
    w: np.ndarray

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def prefill_instance(*, seed: int, layer: int, H: int, D: int, window: int, ratio: int,
                     d_idx: int, topk: int, P: int, T: int, sigma_w: float = 1.0,
                     queries=None) -> PrefillInstance:
    """Draw the inputs of one prefill chunk.  `queries`, if given, is a (q, q_idx) pair
    drawn once elsewhere (several layers fed the same chunk of queries); q_idx is
    dropped on a layer without an indexer."""
    # enough prefix tokens for the raw window and for the compressor's open block
    n_prior = min(P, max(window - 1, P % ratio if ratio > 0 else 0))
    n_given = P // ratio if ratio > 0 else 0
    n_vis_end = (P + T) // ratio if ratio > 0 else 0
    if queries is None:
        q = normal_f16(seed, layer, T_Q, (T, H, D))
        q_idx = normal_f16(seed, layer, T_QIDX, (T, d_idx) if topk > 0 else (T, 0))
    else:
        q, q_idx = queries
        q_idx = q_idx if topk > 0 else np.zeros((T, 0), np.float16)
    return PrefillInstance(
        H=H, D=D, window=window, ratio=ratio, d_idx=d_idx, topk=topk, P=P, T=T, n_prior=n_prior,
        raw_k=normal_f16(seed, layer, T_KRAW, (n_prior + T, D)),
        raw_v=normal_f16(seed, layer, T_VRAW, (n_prior + T, D)),
        comp_k=normal_f16(seed, layer, T_COMPK, (n_given, D)),
        comp_v=normal_f16(seed, layer, T_COMPV, (n_given, D)),
        kidx=normal_f16(seed, layer, T_KIDX, (n_vis_end if topk > 0 else 0, d_idx)),
        q=q, q_idx=q_idx,
        w=normal_f32(seed, layer, T_W, (D,), sigma_w),
    )


def chunk_queries(seed: int, T: int, H: int, D: int, d_idx: int):
    """One draw of a chunk's attention and indexer queries (stream of layer 0)."""
    return normal_f16(seed, 0, T_Q, (T, H, D)), normal_f16(seed, 0, T_QIDX, (T, d_idx))
