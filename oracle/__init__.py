"""CPU oracle of the compressed sparse MQA attention path (fp64, plain C).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path never imports this
package, and this package never imports the product (it takes plain numpy
arrays, or any object with the documented instance fields).

The arithmetic lives in ds4a_oracle.c; this module compiles it with gcc when
the shared object is missing or stale, widens fp16 inputs to double (exact),
and composes the C functions into one decode step or one prefill chunk in the
order the "DS4 (DwarfStar 4)" page, Key Techniques, "KV attention compression"
gives: compressor append, then indexer top-k, then one softmax over the raw
window and the kept compressed rows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds4a_oracle.c")
_LIB = os.path.join(_HERE, "libds4a_oracle.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)
_L = ctypes.c_long


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, -O2, no vectorisation flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.orc_layer_ratio.argtypes = [ctypes.c_int]
        L.orc_layer_topk.argtypes = [ctypes.c_int]
        L.orc_rows_visible.argtypes = [_L, ctypes.c_int]
        L.orc_rows_visible.restype = _L
        L.orc_pool_block.argtypes = [_D, _D, ctypes.c_int, ctypes.c_int, _D, _D, _D]
        L.orc_pool_block.restype = None
        L.orc_compress_range.argtypes = [_D, _D, _L, _L, ctypes.c_int, _D, ctypes.c_int, _L, _L, _D, _D]
        L.orc_compress_range.restype = _L
        L.orc_pool_block_keys.argtypes = [_D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int, _D, _D]
        L.orc_pool_block_keys.restype = None
        L.orc_compress_range_keys.argtypes = [_D, _D, _L, _L, ctypes.c_int, ctypes.c_int, _D, ctypes.c_int, _L, _L,
                                              _D]
        L.orc_compress_range_keys.restype = _L
        L.orc_index_scores.argtypes = [_D, _D, _L, ctypes.c_int, _D]
        L.orc_index_scores.restype = None
        L.orc_topk.argtypes = [_D, _L, ctypes.c_int, _I]
        L.orc_indexer.argtypes = [_D, ctypes.c_int, _D, _L, ctypes.c_int, _L, ctypes.c_int,
                                  ctypes.c_int, _I, _I]
        L.orc_indexer.restype = None
        L.orc_attend.argtypes = [_D, ctypes.c_int, ctypes.c_int, ctypes.c_double, _D, _D, _L, _D]
        L.orc_attend.restype = None
        L.orc_decode_attend.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, _D, _L,
                                        ctypes.c_int, _D, _D, _L, _L, _D, _D, _I, _L, _D]
        L.orc_prefill_attend.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                         _D, _D, _D, _L, ctypes.c_int, _D, _D, _I, ctypes.c_int,
                                         _L, ctypes.c_int, _D]
        _lib = L
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.float64)


def _dp(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _ip(a):
    return None if a is None else a.ctypes.data_as(_I)


# ---- single functions ------------------------------------------------------

def layer_ratio(layer: int) -> int:
    return lib().orc_layer_ratio(layer)


def layer_topk(layer: int) -> int:
    return lib().orc_layer_topk(layer)


def rows_visible(p: int, r: int) -> int:
    return lib().orc_rows_visible(p, r)


def pool_block(k, v, w):
    k, v, w = _f64(k), _f64(v), _f64(w)
    n, D = k.shape
    ok, ov = np.zeros(D), np.zeros(D)
    lib().orc_pool_block(_dp(k), _dp(v), n, D, _dp(w), _dp(ok), _dp(ov))
    return ok, ov


def compress_range(raw_k, raw_v, raw_pos0: int, w, r: int, b0: int, b1: int):
    """Pooled rows b0..b1-1 (float64 [b1-b0, D] each) from raw tokens at positions raw_pos0.."""
    raw_k, raw_v, w = _f64(raw_k), _f64(raw_v), _f64(w)
    n_raw, D = raw_k.shape
    ok = np.zeros((max(b1 - b0, 0), D))
    ov = np.zeros((max(b1 - b0, 0), D))
    rc = lib().orc_compress_range(_dp(raw_k), _dp(raw_v), raw_pos0, n_raw, D, _dp(w), r, b0, b1,
                                  _dp(ok), _dp(ov))
    if rc < 0:
        raise ValueError("compress_range: a block reaches outside the raw rows given")
    return ok, ov


def pool_block_keys(k, ki, w):
    """Pooled indexer key of one block: the block's softmax weights of w . k_t applied
    to the tokens' indexer keys ki [n, DI]."""
    k, ki, w = _f64(k), _f64(ki), _f64(w)
    n, D = k.shape
    DI = ki.shape[1]
    out = np.zeros(DI)
    lib().orc_pool_block_keys(_dp(k), _dp(ki), n, D, DI, _dp(w), _dp(out))
    return out


def compress_range_keys(raw_k, raw_ki, raw_pos0: int, w, r: int, b0: int, b1: int):
    """Pooled indexer keys of blocks b0..b1-1 (float64 [b1-b0, DI]) from the raw tokens'
    K rows and indexer keys at positions raw_pos0.."""
    raw_k, raw_ki, w = _f64(raw_k), _f64(raw_ki), _f64(w)
    n_raw, D = raw_k.shape
    DI = raw_ki.shape[1]
    out = np.zeros((max(b1 - b0, 0), DI))
    rc = lib().orc_compress_range_keys(_dp(raw_k), _dp(raw_ki), raw_pos0, n_raw, D, DI, _dp(w), r, b0, b1,
                                       _dp(out))
    if rc < 0:
        raise ValueError("compress_range_keys: a block reaches outside the raw rows given")
    return out


def index_scores(q, kidx):
    q, kidx = _f64(q), _f64(kidx)
    n, d = kidx.shape
    out = np.zeros(n)
    lib().orc_index_scores(_dp(q), _dp(kidx), n, d, _dp(out))
    return out


def topk(scores, k: int):
    s = _f64(scores)
    out = np.full(max(k, 1), -1, dtype=np.int32)
    m = lib().orc_topk(_dp(s), s.shape[0], k, _ip(out))
    return out[:m]


def indexer(q_idx, kidx, q_pos0: int, ratio: int, k: int):
    """Per-query top-k: returns (idx [n_q, k] int32 ascending, -1 padded; n [n_q])."""
    q_idx, kidx = _f64(np.atleast_2d(q_idx)), _f64(kidx)
    n_q, d = q_idx.shape
    out = np.full((n_q, k), -1, dtype=np.int32)
    out_n = np.zeros(n_q, dtype=np.int32)
    lib().orc_indexer(_dp(q_idx), n_q, _dp(kidx), kidx.shape[0], d, q_pos0, ratio, k,
                      _ip(out), _ip(out_n))
    return out, out_n


def attend(q, K, V, scale: float):
    q, K, V = _f64(q), _f64(K), _f64(V)
    H, D = q.shape
    out = np.zeros((H, D))
    lib().orc_attend(_dp(q), H, D, scale, _dp(K), _dp(V), K.shape[0], _dp(out))
    return out


def decode_attend(q, p: int, window: int, raw_k, raw_v, raw_pos0: int, comp_k, comp_v,
                  sel, n_sel: int, scale: float):
    q, raw_k, raw_v = _f64(q), _f64(raw_k), _f64(raw_v)
    H, D = q.shape
    comp_k = _f64(comp_k).reshape(-1, D) if comp_k is not None else np.zeros((0, D))
    comp_v = _f64(comp_v).reshape(-1, D) if comp_v is not None else np.zeros((0, D))
    sel_a = None if sel is None else np.ascontiguousarray(sel, dtype=np.int32)
    out = np.zeros((H, D))
    rc = lib().orc_decode_attend(H, D, scale, _dp(q), p, window, _dp(raw_k), _dp(raw_v),
                                 raw_pos0, raw_k.shape[0], _dp(comp_k), _dp(comp_v),
                                 _ip(sel_a), n_sel, _dp(out))
    if rc != 0:
        raise ValueError("decode_attend: raw rows do not cover the window")
    return out


def prefill_attend(q, raw_k, raw_v, n_prior: int, window: int, comp_k, comp_v, sel,
                   q_pos0: int, ratio: int, scale: float):
    q, raw_k, raw_v = _f64(q), _f64(raw_k), _f64(raw_v)
    T, H, D = q.shape
    comp_k = _f64(comp_k).reshape(-1, D) if comp_k is not None else np.zeros((0, D))
    comp_v = _f64(comp_v).reshape(-1, D) if comp_v is not None else np.zeros((0, D))
    sel_a = None if sel is None else np.ascontiguousarray(sel, dtype=np.int32)
    k_stride = 0 if sel_a is None else sel_a.shape[1]
    out = np.zeros((T, H, D))
    rc = lib().orc_prefill_attend(T, H, D, scale, _dp(q), _dp(raw_k), _dp(raw_v), n_prior, window,
                                  _dp(comp_k), _dp(comp_v), _ip(sel_a), k_stride, q_pos0, ratio,
                                  _dp(out))
    if rc != 0:
        raise ValueError("prefill_attend: raw rows do not cover a window")
    return out


# ---- composed path: one decode step, one prefill chunk ----------------------

def decode_step(inst) -> dict:
    """Oracle of one decode step of one layer at position inst.p.

    Order: the current token enters the compressor (a block it completes becomes
    visible: append-then-attend), the indexer ranks the visible rows, then one
    softmax runs over the raw window and the kept (or all) compressed rows.  With
    per-token indexer keys (inst.kidx_tok), rows past the given keys are ranked
    by the keys pooled from their tokens' keys.
    Returns out [H, D] float64, sel (ascending kept rows, or None), the pooled
    rows (float64) and the number of visible rows.
    """
    p, r, D = inst.p, inst.ratio, inst.D
    sel = None
    ck = cv = None
    n_vis = 0
    if r > 0:
        n_vis = rows_visible(p, r)
        if inst.pooled_history:
            ck, cv = compress_range(inst.raw_k, inst.raw_v, 0, inst.w, r, 0, n_vis)
        else:
            n_given = inst.comp_k.shape[0]
            ck, cv = _f64(inst.comp_k).reshape(-1, D), _f64(inst.comp_v).reshape(-1, D)
            if n_vis > n_given:
                nk, nv = compress_range(inst.raw_k, inst.raw_v, inst.raw_pos0, inst.w, r, n_given, n_vis)
                ck, cv = np.concatenate([ck, nk]), np.concatenate([cv, nv])
        if inst.topk > 0:
            kidx = inst.kidx
            ki_tok = getattr(inst, "kidx_tok", None)
            if ki_tok is not None and n_vis > kidx.shape[0]:
                # pooled keys: the rows past the given ones take the keys the compressor
                # pools from their tokens' indexer keys, with the same weights as K and V
                pk = compress_range_keys(inst.raw_k, ki_tok, inst.raw_pos0, inst.w, r, kidx.shape[0], n_vis)
                kidx = np.concatenate([_f64(kidx).reshape(-1, pk.shape[1]), pk])
            idx, n = indexer(inst.q_idx[None, :], kidx, p, r, inst.topk)
            sel = idx[0, : n[0]]
    n_sel = (len(sel) if sel is not None else n_vis)
    out = decode_attend(inst.q, p, inst.window, inst.raw_k, inst.raw_v, inst.raw_pos0,
                        ck, cv, sel, n_sel, inst.scale)
    return {"out": out, "sel": sel, "comp_k": ck, "comp_v": cv, "n_vis": n_vis}


def prefill_chunk(inst) -> dict:
    """Oracle of one prefill chunk: pool the blocks the chunk completes, rank the
    rows visible to each query, then per query one softmax over its raw window and
    its kept (or all visible) compressed rows.  Returns out [T, H, D] float64,
    sel [T, k] (-1 padded) or None, sel_n [T] or None, and the new pooled rows."""
    P, T, r, D = inst.P, inst.T, inst.ratio, inst.D
    raw_pos0 = P - inst.n_prior
    sel = sel_n = None
    ck = cv = nk = nv = None
    if r > 0:
        b0, b1 = P // r, (P + T) // r
        nk, nv = compress_range(inst.raw_k, inst.raw_v, raw_pos0, inst.w, r, b0, b1)
        ck = np.concatenate([_f64(inst.comp_k).reshape(-1, D), nk])
        cv = np.concatenate([_f64(inst.comp_v).reshape(-1, D), nv])
        if inst.topk > 0:
            sel, sel_n = indexer(inst.q_idx, inst.kidx, P, r, inst.topk)
    out = prefill_attend(inst.q, inst.raw_k, inst.raw_v, inst.n_prior, inst.window, ck, cv, sel,
                         P, r, inst.scale)
    return {"out": out, "sel": sel, "sel_n": sel_n, "new_k": nk, "new_v": nv}
