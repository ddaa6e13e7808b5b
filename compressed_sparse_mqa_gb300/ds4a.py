"""Thin ctypes binding of libds4a.so (include/ds4a.h).

Argument marshalling only: every function takes torch CUDA tensors (the host
inputs and output of ds4a_decode_layer_step: CPU tensors), checks dtype /
contiguity / device, passes raw pointers and the current CUDA stream to the C
entry point of the same name, and raises Ds4aError on a non-zero status.  All arithmetic runs in the library's CUDA kernels.  There is no CPU
fallback: if the library has not been built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libds4a.so")
_lib = None

DS4A_OK = 0
DS4A_ERR_ARG = 1
DS4A_ERR_CAPACITY = 2
DS4A_ERR_UNSUPPORTED = 3
DS4A_ERR_CUDA = 4
DS4A_ERR_TIMEOUT = 5
DS4A_ERR_WORKSPACE = 6
DS4A_ERR_DEVICE_INDEX = 7

EXPORTED = ["ds4a_status_str", "ds4a_last_device_error", "ds4a_compress_append",
            "ds4a_indexer_topk", "ds4a_indexer_workspace_bytes", "ds4a_attn_decode",
            "ds4a_attn_prefill", "ds4a_indexer_topk_compress", "ds4a_compress_attn_decode",
            "ds4a_indexer_topk_noalloc", "ds4a_test_set_wait_limit", "ds4a_compress_append_keys",
            "ds4a_decode_batched_workspace_bytes", "ds4a_indexer_topk_compress_batched", "ds4a_attn_decode_batched",
            "ds4a_compress_attn_decode_batched", "ds4a_probe_gather", "ds4a_decode_layer_step",
            "ds4a_indexer_topk_compress_keys"]


class Ds4aError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} (status {status})")


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libds4a.so is not built ({LIB_PATH}); run compressed_sparse_mqa_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, LL, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float, ctypes.c_size_t
        L.ds4a_status_str.argtypes = [I]
        L.ds4a_status_str.restype = ctypes.c_char_p
        L.ds4a_last_device_error.argtypes = [P]
        L.ds4a_test_set_wait_limit.argtypes = [LL]
        L.ds4a_indexer_topk_noalloc.argtypes = [P, P, LL, I, LL, I, I, P, P, P]
        L.ds4a_compress_append.argtypes = [P, P, I, I, P, I, LL, P, P, P, LL, P]
        L.ds4a_indexer_topk.argtypes = [P, I, P, LL, I, LL, I, I, P, P, P, SZ, P]
        L.ds4a_compress_append_keys.argtypes = [P, P, P, I, I, I, P, I, LL, P, P, P, P, LL, P]
        L.ds4a_probe_gather.argtypes = [P, LL, I, P, LL, P, P]
        L.ds4a_decode_batched_workspace_bytes.argtypes = [I, LL]
        L.ds4a_decode_batched_workspace_bytes.restype = SZ
        L.ds4a_indexer_topk_compress_batched.argtypes = [I, P, P, LL, I, P, I, I, P, P, P, SZ, P, P, I, I, P, P, P, P, P]
        L.ds4a_attn_decode_batched.argtypes = [I, P, I, I, P, P, I, P, P, P, LL, P, I, I, F, P, P]
        L.ds4a_compress_attn_decode_batched.argtypes = [I, P, I, P, P, P, LL, P, I, I, P, P, I, P, F, P, P]
        L.ds4a_indexer_topk_compress.argtypes = [P, P, LL, I, LL, I, I, P, P, P, SZ, P, P, I, P, P, P, P, LL, P]
        L.ds4a_indexer_topk_compress_keys.argtypes = [P, P, LL, I, LL, I, I, P, P, P, SZ, P, P, P, I, P, P, P, P, LL, P]
        L.ds4a_compress_attn_decode.argtypes = [P, P, P, I, LL, P, P, P, LL, P, I, I, P, P, I, F, P, P]
        L.ds4a_indexer_workspace_bytes.argtypes = [I, LL, I]
        L.ds4a_indexer_workspace_bytes.restype = SZ
        L.ds4a_attn_decode.argtypes = [P, I, I, P, P, I, P, P, LL, P, I, F, P, P, SZ, P]
        L.ds4a_attn_prefill.argtypes = [P, I, I, I, P, P, I, I, P, P, LL, P, I, LL, I, F, P, P, SZ, P]
        L.ds4a_decode_layer_step.argtypes = [ctypes.POINTER(DecodeLayerDesc), LL, ctypes.POINTER(DecodeHostInputs),
                                             P, P]
        for name in EXPORTED:
            if name not in ("ds4a_status_str", "ds4a_indexer_workspace_bytes", "ds4a_decode_batched_workspace_bytes"):
                getattr(L, name).restype = I
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().ds4a_status_str(status).decode()


def _check(rc: int, where: str):
    if rc != DS4A_OK:
        raise Ds4aError(rc, where)


def _ptr(t, dtype, name, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def ds4a_last_device_error(stream=None) -> int:
    return lib().ds4a_last_device_error(_stream(stream))


def ds4a_test_set_wait_limit(limit_ns: int):
    """Test hook: decode attention launches enqueued afterwards add a wait that gives up
    after limit_ns and records DS4A_ERR_TIMEOUT (0 turns it off)."""
    _check(lib().ds4a_test_set_wait_limit(int(limit_ns)), "ds4a_test_set_wait_limit")


def ds4a_compress_append(k, v, score_w, ratio: int, pos: int, state, comp_k, comp_v, stream=None):
    """Feed k/v [n_new, D] (fp16) at positions pos.. to the compressor; writes pooled
    rows into comp_k/comp_v [cap, D] and the open block's state [2+2D] (fp32)."""
    n_new, D = k.shape
    if v.shape != k.shape or comp_k.shape != comp_v.shape or comp_k.shape[1] != D:
        raise ValueError("compress_append: shape mismatch")
    if state.numel() < 2 + 2 * D or score_w.numel() != D:
        raise ValueError("compress_append: state / score_w size")
    rc = lib().ds4a_compress_append(_ptr(k, torch.float16, "k"), _ptr(v, torch.float16, "v"), n_new, D,
                                    _ptr(score_w, torch.float32, "score_w"), ratio, pos,
                                    _ptr(state, torch.float32, "state"),
                                    _ptr(comp_k, torch.float16, "comp_k"),
                                    _ptr(comp_v, torch.float16, "comp_v"), comp_k.shape[0], _stream(stream))
    _check(rc, "ds4a_compress_append")


def _marshal_compress_append_keys(k, v, ki, score_w, ratio: int, pos: int, state, comp_k, comp_v, comp_kidx,
                                  stream=None):
    n_new, D = k.shape
    DI = ki.shape[1]
    if v.shape != k.shape or ki.shape[0] != n_new or comp_k.shape != comp_v.shape or comp_k.shape[1] != D:
        raise ValueError("compress_append_keys: shape mismatch")
    if comp_kidx.shape[0] != comp_k.shape[0] or comp_kidx.shape[1] != DI:
        raise ValueError("compress_append_keys: pooled-key rows must match the compressed rows")
    if state.numel() < 2 + 2 * D + DI or score_w.numel() != D:
        raise ValueError("compress_append_keys: state / score_w size")
    return (_ptr(k, torch.float16, "k"), _ptr(v, torch.float16, "v"), _ptr(ki, torch.float16, "ki"), n_new, D, DI,
            _ptr(score_w, torch.float32, "score_w"), ratio, pos, _ptr(state, torch.float32, "state"),
            _ptr(comp_k, torch.float16, "comp_k"), _ptr(comp_v, torch.float16, "comp_v"),
            _ptr(comp_kidx, torch.float16, "comp_kidx"), comp_k.shape[0], _stream(stream))


def ds4a_compress_append_keys(k, v, ki, score_w, ratio: int, pos: int, state, comp_k, comp_v, comp_kidx,
                              stream=None):
    """ds4a_compress_append that also pools the tokens' indexer keys ki [n_new, DI] into
    comp_kidx [cap, DI] with the same weights; state [2 + 2D + DI] fp32."""
    args = _marshal_compress_append_keys(k, v, ki, score_w, ratio, pos, state, comp_k, comp_v, comp_kidx, stream)
    _check(lib().ds4a_compress_append_keys(*args), "ds4a_compress_append_keys")


def _marshal_indexer_topk(q_idx, k_idx, q_pos0: int, ratio: int, k: int, out_idx, out_n, ws, n_rows=None,
                          stream=None):
    q2 = q_idx if q_idx.dim() == 2 else q_idx.view(1, -1)
    n_q, d = q2.shape
    rows = k_idx.shape[0] if n_rows is None else n_rows
    if k_idx.shape[0] < rows or (k_idx.numel() and k_idx.shape[1] != d):
        raise ValueError("indexer_topk: k_idx shape")
    if out_idx.numel() < n_q * k:
        raise ValueError("indexer_topk: out_idx too small")
    return (_ptr(q2, torch.float16, "q_idx"), n_q, _ptr(k_idx, torch.float16, "k_idx") if k_idx.numel() else None,
            rows, d, q_pos0, ratio, k, _ptr(out_idx, torch.int32, "out_idx"),
            _ptr(out_n, torch.int32, "out_n", optional=True), _ptr(ws, torch.uint8, "ws"), ws.numel(),
            _stream(stream))


def ds4a_indexer_workspace_bytes(n_q: int, n_rows: int, k: int) -> int:
    return int(lib().ds4a_indexer_workspace_bytes(n_q, n_rows, k))


def ds4a_indexer_topk(q_idx, k_idx, q_pos0: int, ratio: int, k: int, out_idx, out_n, ws, n_rows=None,
                      stream=None):
    """q_idx [n_q, d] fp16, k_idx [n_rows, d] fp16 -> out_idx [n_q, k] int32 (ascending, -1 pad),
    out_n [n_q] int32 (or None).  ws: uint8 tensor of ds4a_indexer_workspace_bytes bytes."""
    args = _marshal_indexer_topk(q_idx, k_idx, q_pos0, ratio, k, out_idx, out_n, ws, n_rows, stream)
    _check(lib().ds4a_indexer_topk(*args), "ds4a_indexer_topk")


def _marshal_indexer_topk_compress(q_idx, k_idx, q_pos: int, ratio: int, k: int, out_idx, out_n, ws, k_new, v_new,
                                   score_w, state, comp_k, comp_v, n_rows=None, stream=None):
    q2 = q_idx if q_idx.dim() == 2 else q_idx.view(1, -1)
    if q2.shape[0] != 1:
        raise ValueError("indexer_topk_compress: one query")
    d = q2.shape[1]
    rows = k_idx.shape[0] if n_rows is None else n_rows
    if k_idx.shape[0] < rows or (k_idx.numel() and k_idx.shape[1] != d):
        raise ValueError("indexer_topk_compress: k_idx shape")
    if out_idx.numel() < k:
        raise ValueError("indexer_topk_compress: out_idx too small")
    n_new, D = k_new.shape
    if n_new != 1 or v_new.shape != k_new.shape or comp_k.shape != comp_v.shape or comp_k.shape[1] != D:
        raise ValueError("indexer_topk_compress: token / compressed-row shapes")
    if state.numel() < 2 + 2 * D or score_w.numel() != D:
        raise ValueError("indexer_topk_compress: state / score_w size")
    return (_ptr(q2, torch.float16, "q_idx"), _ptr(k_idx, torch.float16, "k_idx") if k_idx.numel() else None, rows,
            d, q_pos, ratio, k, _ptr(out_idx, torch.int32, "out_idx"), _ptr(out_n, torch.int32, "out_n", optional=True),
            _ptr(ws, torch.uint8, "ws"), ws.numel(), _ptr(k_new, torch.float16, "k_new"),
            _ptr(v_new, torch.float16, "v_new"), D, _ptr(score_w, torch.float32, "score_w"),
            _ptr(state, torch.float32, "state"), _ptr(comp_k, torch.float16, "comp_k"),
            _ptr(comp_v, torch.float16, "comp_v"), comp_k.shape[0], _stream(stream))


def ds4a_indexer_topk_compress(q_idx, k_idx, q_pos: int, ratio: int, k: int, out_idx, out_n, ws, k_new, v_new,
                               score_w, state, comp_k, comp_v, n_rows=None, stream=None):
    """ds4a_indexer_topk for one query at q_pos (q_idx [d] or [1, d]) and
    ds4a_compress_append of that position's token (k_new, v_new [1, D] fp16), in one
    launch; arguments as the two calls."""
    args = _marshal_indexer_topk_compress(q_idx, k_idx, q_pos, ratio, k, out_idx, out_n, ws, k_new, v_new, score_w,
                                          state, comp_k, comp_v, n_rows, stream)
    _check(lib().ds4a_indexer_topk_compress(*args), "ds4a_indexer_topk_compress")


def _marshal_indexer_topk_compress_keys(q_idx, k_idx, q_pos: int, ratio: int, k: int, out_idx, out_n, ws, k_new,
                                        v_new, k_idx_tok, score_w, state, comp_k, comp_v, n_rows=None, stream=None):
    args = list(_marshal_indexer_topk_compress(q_idx, k_idx, q_pos, ratio, k, out_idx, out_n, ws, k_new, v_new,
                                               score_w, state, comp_k, comp_v, n_rows, stream))
    d = args[3]
    if k_idx_tok is None or k_idx_tok.numel() != d or k_idx.numel() == 0:
        raise ValueError("indexer_topk_compress_keys: k_idx_tok [d_idx] and k_idx rows are required")
    # (q_idx, k_idx, rows, d, q_pos, ratio, k, out_idx, out_n, ws, ws_bytes, k_new, v_new, | k_idx_tok |, D, ...)
    args.insert(13, _ptr(k_idx_tok, torch.float16, "k_idx_tok"))
    return tuple(args)


def ds4a_indexer_topk_compress_keys(q_idx, k_idx, q_pos: int, ratio: int, k: int, out_idx, out_n, ws, k_new, v_new,
                                    k_idx_tok, score_w, state, comp_k, comp_v, n_rows=None, stream=None):
    """ds4a_compress_append_keys of the token at q_pos (k_new, v_new [1, D], k_idx_tok [d]
    or [1, d]) into comp rows and the indexer keys k_idx, and ds4a_indexer_topk of the
    step's query over k_idx, in one launch."""
    args = _marshal_indexer_topk_compress_keys(q_idx, k_idx, q_pos, ratio, k, out_idx, out_n, ws, k_new, v_new,
                                               k_idx_tok, score_w, state, comp_k, comp_v, n_rows, stream)
    _check(lib().ds4a_indexer_topk_compress_keys(*args), "ds4a_indexer_topk_compress_keys")


def _marshal_compress_attn_decode(k_new, v_new, score_w, ratio: int, pos: int, state, comp_k, comp_v, q, win_k,
                                  win_v, scale: float, out, stream=None):
    H, D = q.shape
    if k_new.shape != (1, D) or v_new.shape != (1, D) or comp_k.shape != comp_v.shape or comp_k.shape[1] != D:
        raise ValueError("compress_attn_decode: token / compressed-row shapes")
    if win_k.shape != win_v.shape or win_k.shape[1] != D or out.shape != q.shape:
        raise ValueError("compress_attn_decode: window / output shapes")
    if state.numel() < 2 + 2 * D or score_w.numel() != D:
        raise ValueError("compress_attn_decode: state / score_w size")
    return (_ptr(k_new, torch.float16, "k_new"), _ptr(v_new, torch.float16, "v_new"),
            _ptr(score_w, torch.float32, "score_w"), ratio, pos, _ptr(state, torch.float32, "state"),
            _ptr(comp_k, torch.float16, "comp_k"), _ptr(comp_v, torch.float16, "comp_v"), comp_k.shape[0],
            _ptr(q, torch.float16, "q"), H, D, _ptr(win_k, torch.float16, "win_k"), _ptr(win_v, torch.float16, "win_v"),
            win_k.shape[0], scale, _ptr(out, torch.float16, "out"), _stream(stream))


def ds4a_compress_attn_decode(k_new, v_new, score_w, ratio: int, pos: int, state, comp_k, comp_v, q, win_k, win_v,
                              scale: float, out, stream=None):
    """ds4a_compress_append of the token at pos (k_new, v_new [1, D] fp16) and
    ds4a_attn_decode over the window and every visible compressed row, in one launch;
    arguments as the two calls."""
    args = _marshal_compress_attn_decode(k_new, v_new, score_w, ratio, pos, state, comp_k, comp_v, q, win_k, win_v,
                                         scale, out, stream)
    _check(lib().ds4a_compress_attn_decode(*args), "ds4a_compress_attn_decode")


def _marshal_attn_decode(q, win_k, win_v, comp_k, comp_v, sel, n_sel: int, scale: float, out, stream=None):
    H, D = q.shape
    n_win = win_k.shape[0]
    n_comp = 0 if comp_k is None else comp_k.shape[0]
    return (_ptr(q, torch.float16, "q"), H, D, _ptr(win_k, torch.float16, "win_k"),
            _ptr(win_v, torch.float16, "win_v"), n_win,
            _ptr(comp_k, torch.float16, "comp_k", optional=True),
            _ptr(comp_v, torch.float16, "comp_v", optional=True), n_comp,
            _ptr(sel, torch.int32, "sel", optional=True), n_sel, scale,
            _ptr(out, torch.float16, "out"), None, 0, _stream(stream))


def ds4a_attn_decode(q, win_k, win_v, comp_k, comp_v, sel, n_sel: int, scale: float, out, stream=None):
    """q [H, D] fp16; window rows win_k/win_v [n_win, D]; comp rows [n_comp, D]; sel int32 [>= n_sel]
    or None (rows 0..n_sel-1); out [H, D] fp16."""
    args = _marshal_attn_decode(q, win_k, win_v, comp_k, comp_v, sel, n_sel, scale, out, stream)
    _check(lib().ds4a_attn_decode(*args), "ds4a_attn_decode")


def ds4a_attn_prefill(q, raw_k, raw_v, n_prior: int, window: int, comp_k, comp_v, sel, q_pos0: int,
                      ratio: int, scale: float, out, stream=None):
    """q [T, H, D] fp16; raw rows [n_prior + T, D] for positions q_pos0-n_prior..; comp rows
    [n_comp, D] (or None); sel [T, k_stride] int32 or None; out [T, H, D] fp16."""
    T, H, D = q.shape
    n_comp = 0 if comp_k is None else comp_k.shape[0]
    k_stride = 0 if sel is None else sel.shape[1]
    rc = lib().ds4a_attn_prefill(_ptr(q, torch.float16, "q"), T, H, D, _ptr(raw_k, torch.float16, "raw_k"),
                                 _ptr(raw_v, torch.float16, "raw_v"), n_prior, window,
                                 _ptr(comp_k, torch.float16, "comp_k", optional=True),
                                 _ptr(comp_v, torch.float16, "comp_v", optional=True), n_comp,
                                 _ptr(sel, torch.int32, "sel", optional=True), k_stride, q_pos0, ratio, scale,
                                 _ptr(out, torch.float16, "out"), None, 0, _stream(stream))
    _check(rc, "ds4a_attn_prefill")


def ds4a_probe_gather(table, idx, sink, stream=None):
    """Measurement call: gather rows table[idx] ([n, D] fp16, idx int32) into shared memory;
    sink: a one-element int32 device tensor that receives one word of the result."""
    rc = lib().ds4a_probe_gather(_ptr(table, torch.float16, "table"), table.shape[0], table.shape[1],
                                 _ptr(idx, torch.int32, "idx"), idx.numel(), _ptr(sink, torch.int32, "sink"),
                                 _stream(stream))
    _check(rc, "ds4a_probe_gather")


def ds4a_decode_batched_workspace_bytes(B: int, cap: int) -> int:
    return int(lib().ds4a_decode_batched_workspace_bytes(B, cap))


def _marshal_indexer_topk_compress_batched(q_idx, k_idx, pos, ratio: int, k: int, out_idx, out_n, ws, ring_k,
                                           ring_v, score_w, state, comp_k, comp_v, stream=None):
    B, cap, d = k_idx.shape
    _, W, D = ring_k.shape
    if q_idx.shape != (B, d) or pos.shape != (B,) or out_idx.shape[0] != B or out_idx.shape[1] < k:
        raise ValueError("indexer_topk_compress_batched: query / position / output shapes")
    if ring_v.shape != ring_k.shape or ring_k.shape[0] != B or comp_k.shape != (B, cap, D) or comp_v.shape != comp_k.shape:
        raise ValueError("indexer_topk_compress_batched: ring / compressed-row shapes")
    if state.shape != (B, 2 + 2 * D) or score_w.numel() != D or out_idx.shape[1] != k:
        raise ValueError("indexer_topk_compress_batched: state / score_w / out_idx shapes")
    return (B, _ptr(q_idx, torch.float16, "q_idx"), _ptr(k_idx, torch.float16, "k_idx"), cap, d,
            _ptr(pos, torch.int64, "pos"), ratio, k, _ptr(out_idx, torch.int32, "out_idx"),
            _ptr(out_n, torch.int32, "out_n", optional=True), _ptr(ws, torch.uint8, "ws"), ws.numel(),
            _ptr(ring_k, torch.float16, "ring_k"), _ptr(ring_v, torch.float16, "ring_v"), W, D,
            _ptr(score_w, torch.float32, "score_w"), _ptr(state, torch.float32, "state"),
            _ptr(comp_k, torch.float16, "comp_k"), _ptr(comp_v, torch.float16, "comp_v"), _stream(stream))


def ds4a_indexer_topk_compress_batched(q_idx, k_idx, pos, ratio: int, k: int, out_idx, out_n, ws, ring_k, ring_v,
                                       score_w, state, comp_k, comp_v, stream=None):
    """B sessions: q_idx [B, d], k_idx [B, cap, d], pos int64 [B] (device), out_idx [B, k],
    rings [B, W, D], state [B, 2 + 2D], comp rows [B, cap, D]."""
    args = _marshal_indexer_topk_compress_batched(q_idx, k_idx, pos, ratio, k, out_idx, out_n, ws, ring_k, ring_v,
                                                  score_w, state, comp_k, comp_v, stream)
    _check(lib().ds4a_indexer_topk_compress_batched(*args), "ds4a_indexer_topk_compress_batched")


def _marshal_attn_decode_batched(q, ring_k, ring_v, pos, comp_k, comp_v, sel, ratio: int, scale: float, out,
                                 stream=None):
    B, H, D = q.shape
    W = ring_k.shape[1]
    cap = 0 if comp_k is None else comp_k.shape[1]
    if ring_k.shape != (B, W, D) or ring_v.shape != ring_k.shape or pos.shape != (B,) or out.shape != q.shape:
        raise ValueError("attn_decode_batched: shapes")
    if comp_k is not None and (comp_k.shape != (B, cap, D) or comp_v.shape != comp_k.shape):
        raise ValueError("attn_decode_batched: compressed-row shapes")
    n_sel = 0 if sel is None else sel.shape[1]
    if sel is not None and sel.shape[0] != B:
        raise ValueError("attn_decode_batched: sel shape")
    return (B, _ptr(q, torch.float16, "q"), H, D, _ptr(ring_k, torch.float16, "ring_k"),
            _ptr(ring_v, torch.float16, "ring_v"), W, _ptr(pos, torch.int64, "pos"),
            _ptr(comp_k, torch.float16, "comp_k", optional=True), _ptr(comp_v, torch.float16, "comp_v", optional=True),
            cap, _ptr(sel, torch.int32, "sel", optional=True), n_sel, ratio, scale, _ptr(out, torch.float16, "out"),
            _stream(stream))


def ds4a_attn_decode_batched(q, ring_k, ring_v, pos, comp_k, comp_v, sel, ratio: int, scale: float, out,
                             stream=None):
    """B sessions: q [B, H, D], rings [B, W, D], pos int64 [B] (device), comp rows [B, cap, D] (or
    None), sel [B, n] int32 or None (every visible row), out [B, H, D]."""
    args = _marshal_attn_decode_batched(q, ring_k, ring_v, pos, comp_k, comp_v, sel, ratio, scale, out, stream)
    _check(lib().ds4a_attn_decode_batched(*args), "ds4a_attn_decode_batched")


def _marshal_compress_attn_decode_batched(score_w, ratio: int, state, comp_k, comp_v, q, ring_k, ring_v, pos,
                                          scale: float, out, stream=None):
    B, H, D = q.shape
    W = ring_k.shape[1]
    cap = comp_k.shape[1]
    if ring_k.shape != (B, W, D) or ring_v.shape != ring_k.shape or pos.shape != (B,) or out.shape != q.shape:
        raise ValueError("compress_attn_decode_batched: shapes")
    if comp_k.shape != (B, cap, D) or comp_v.shape != comp_k.shape or state.shape != (B, 2 + 2 * D):
        raise ValueError("compress_attn_decode_batched: compressed-row / state shapes")
    return (B, _ptr(score_w, torch.float32, "score_w"), ratio, _ptr(state, torch.float32, "state"),
            _ptr(comp_k, torch.float16, "comp_k"), _ptr(comp_v, torch.float16, "comp_v"), cap,
            _ptr(q, torch.float16, "q"), H, D, _ptr(ring_k, torch.float16, "ring_k"),
            _ptr(ring_v, torch.float16, "ring_v"), W, _ptr(pos, torch.int64, "pos"), scale,
            _ptr(out, torch.float16, "out"), _stream(stream))


def ds4a_compress_attn_decode_batched(score_w, ratio: int, state, comp_k, comp_v, q, ring_k, ring_v, pos,
                                      scale: float, out, stream=None):
    """B sessions of a layer that attends every row: each session's compressor update
    and attention in one launch."""
    args = _marshal_compress_attn_decode_batched(score_w, ratio, state, comp_k, comp_v, q, ring_k, ring_v, pos,
                                                 scale, out, stream)
    _check(lib().ds4a_compress_attn_decode_batched(*args), "ds4a_compress_attn_decode_batched")


# ---- one decode step of one layer from host memory --------------------------------------------

class DecodeLayerDesc(ctypes.Structure):
    """ds4a_decode_layer_t: a layer's persistent device arrays (see decode_layer_desc)."""
    _fields_ = [("H", ctypes.c_int), ("D", ctypes.c_int), ("W", ctypes.c_int), ("ratio", ctypes.c_int),
                ("topk", ctypes.c_int), ("d_idx", ctypes.c_int), ("pooled_keys", ctypes.c_int),
                ("scale", ctypes.c_float), ("cap", ctypes.c_longlong),
                ("ring_k", ctypes.c_void_p), ("ring_v", ctypes.c_void_p), ("score_w", ctypes.c_void_p),
                ("state", ctypes.c_void_p), ("comp_k", ctypes.c_void_p), ("comp_v", ctypes.c_void_p),
                ("k_idx", ctypes.c_void_p), ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p),
                ("k_idx_tok", ctypes.c_void_p), ("out_idx", ctypes.c_void_p), ("out_n", ctypes.c_void_p),
                ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t), ("out", ctypes.c_void_p)]


class DecodeHostInputs(ctypes.Structure):
    """ds4a_decode_host_inputs_t: host pointers of one step's inputs (None: already on the device)."""
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p),
                ("k_idx_row", ctypes.c_void_p), ("k_idx_tok", ctypes.c_void_p)]


def _host_ptr(t, dtype, numel, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) torch tensor")
    if t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous {dtype} tensor")
    if t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")
    return t.data_ptr()


def decode_layer_desc(ring_k, ring_v, q, out, scale: float, ratio: int = 0, score_w=None, state=None, comp_k=None,
                      comp_v=None, topk: int = 0, k_idx=None, q_idx=None, out_idx=None, out_n=None, ws=None,
                      k_idx_tok=None) -> DecodeLayerDesc:
    """The ds4a_decode_layer_t of a layer's device tensors: ring_k, ring_v [W, D], q and
    out [H, D] fp16; on a compressing layer score_w [D] and state float, comp_k, comp_v
    [cap, D] fp16; on an indexer layer k_idx [>= cap, d_idx], q_idx [d_idx], out_idx
    [topk] int32, out_n or None, ws uint8, and k_idx_tok [d_idx] when the compressor
    pools the indexer keys.  The descriptor holds the tensors' addresses: keep them alive."""
    H, D = q.shape
    W = ring_k.shape[0]
    if ring_k.shape != (W, D) or ring_v.shape != (W, D) or out.shape != q.shape:
        raise ValueError("decode_layer_desc: ring / output shapes")
    desc = DecodeLayerDesc(H=H, D=D, W=W, ratio=ratio, topk=topk, scale=scale,
                           ring_k=_ptr(ring_k, torch.float16, "ring_k"), ring_v=_ptr(ring_v, torch.float16, "ring_v"),
                           q=_ptr(q, torch.float16, "q"), out=_ptr(out, torch.float16, "out"))
    if ratio:
        if comp_k.shape != comp_v.shape or comp_k.shape[1] != D or score_w.numel() != D:
            raise ValueError("decode_layer_desc: compressed-row / score_w shapes")
        desc.cap = comp_k.shape[0]
        desc.score_w = _ptr(score_w, torch.float32, "score_w")
        desc.state = _ptr(state, torch.float32, "state")
        desc.comp_k = _ptr(comp_k, torch.float16, "comp_k")
        desc.comp_v = _ptr(comp_v, torch.float16, "comp_v")
    if topk:
        d_idx = q_idx.numel()
        if k_idx.shape[0] < desc.cap or k_idx.shape[1] != d_idx or out_idx.numel() < topk:
            raise ValueError("decode_layer_desc: indexer shapes")
        desc.d_idx = d_idx
        desc.k_idx = _ptr(k_idx, torch.float16, "k_idx")
        desc.q_idx = _ptr(q_idx, torch.float16, "q_idx")
        desc.out_idx = _ptr(out_idx, torch.int32, "out_idx")
        desc.out_n = _ptr(out_n, torch.int32, "out_n", optional=True)
        desc.ws = _ptr(ws, torch.uint8, "ws")
        desc.ws_bytes = ws.numel()
        if k_idx_tok is not None:
            desc.pooled_keys = 1
            desc.k_idx_tok = _ptr(k_idx_tok, torch.float16, "k_idx_tok")
    return desc


def _marshal_decode_layer_step(desc: DecodeLayerDesc, pos: int, k=None, v=None, q=None, q_idx=None, k_idx_row=None,
                               k_idx_tok=None, out_host=None, stream=None):
    D, d = desc.D, desc.d_idx
    f16 = torch.float16
    ins = DecodeHostInputs(k=_host_ptr(k, f16, D, "k"), v=_host_ptr(v, f16, D, "v"),
                           q=_host_ptr(q, f16, desc.H * D, "q"), q_idx=_host_ptr(q_idx, f16, d, "q_idx"),
                           k_idx_row=_host_ptr(k_idx_row, f16, d, "k_idx_row"),
                           k_idx_tok=_host_ptr(k_idx_tok, f16, d, "k_idx_tok"))
    return (ctypes.byref(desc), pos, ctypes.byref(ins), _host_ptr(out_host, f16, desc.H * D, "out_host"),
            _stream(stream))


def ds4a_decode_layer_step(desc: DecodeLayerDesc, pos: int, k=None, v=None, q=None, q_idx=None, k_idx_row=None,
                           k_idx_tok=None, out_host=None, stream=None):
    """The decode step of the token at pos from host tensors (contiguous fp16 CPU
    tensors, page-locked for asynchronous copies; None: that input is already on the
    device); the output is copied into out_host ([H, D] fp16, CPU) and the stream waited
    for, unless out_host is None."""
    args = _marshal_decode_layer_step(desc, pos, k, v, q, q_idx, k_idx_row, k_idx_tok, out_host, stream)
    _check(lib().ds4a_decode_layer_step(*args), "ds4a_decode_layer_step")


_MARSHAL = {"ds4a_attn_decode": _marshal_attn_decode,
            "ds4a_indexer_topk_compress_batched": _marshal_indexer_topk_compress_batched,
            "ds4a_attn_decode_batched": _marshal_attn_decode_batched,
            "ds4a_compress_attn_decode_batched": _marshal_compress_attn_decode_batched,
            "ds4a_indexer_topk": _marshal_indexer_topk,
            "ds4a_compress_append_keys": _marshal_compress_append_keys,
            "ds4a_compress_attn_decode": _marshal_compress_attn_decode,
            "ds4a_indexer_topk_compress": _marshal_indexer_topk_compress,
            "ds4a_decode_layer_step": _marshal_decode_layer_step,
            "ds4a_indexer_topk_compress_keys": _marshal_indexer_topk_compress_keys}


def bind(name: str, *args, **kwargs):
    """The C call that the binding function `name` makes for these arguments,
    marshalled once: returns a zero-argument callable that repeats exactly that call
    (the same device buffers and stream) and raises Ds4aError on a non-zero status.
    For a step repeated on persistent tensors (the per-call Python checks run once)."""
    f = getattr(lib(), name)
    cargs = tuple(_MARSHAL[name](*args, **kwargs))

    def call():
        rc = f(*cargs)
        if rc != DS4A_OK:
            raise Ds4aError(rc, name)
    return call
