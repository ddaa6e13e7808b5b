"""Consecutive calls issued back to back on one stream, with no host sync between
them: decode steps of one layer that share the kept-row list, the indexer
workspace and the compressor state, and prefill chunks that follow one another.

Each kernel starts the work that reads only the caller's inputs before it waits
for the previous kernel (programmatic dependent launch), and writes after the
wait.  These tests check every step of such a sequence against the oracle, run
step by step on the host, so that a write that overtook a read of the previous
call would show up as a wrong output.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import ds4a, synth
from parity import check_out, check_sel

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("ratio,topk,fused", [(4, 16, False), (4, 16, True), (128, 0, False), (128, 0, True)])
def test_decode_steps_back_to_back(ratio, topk, fused):
    H, D, W, d_idx, seed = 8, 64, 32, 32, 5
    p0, S = 200 if ratio == 4 else 1020, 12
    p_end = p0 + S                              # positions p0 .. p0+S-1 are decoded
    raw_k = synth.normal_f16(seed, 1, synth.T_KRAW, (p_end, D))
    raw_v = synth.normal_f16(seed, 1, synth.T_VRAW, (p_end, D))
    w = synth.normal_f32(seed, 1, synth.T_W, (D,), 1.0 / math.sqrt(D))
    n_rows = p_end // ratio                     # every row the sequence completes
    kidx = synth.normal_f16(seed, 1, synth.T_KIDX, (max(n_rows, 1), d_idx))
    q = synth.normal_f16(seed, 1, synth.T_Q, (S, H, D))
    q_idx = synth.normal_f16(seed, 1, synth.T_QIDX, (S, d_idx))
    scale = 1.0 / math.sqrt(D)

    # device state at p0: rows of the blocks complete before p0 pooled by the GPU
    # compressor, which then holds the open block's state
    comp_k = torch.zeros(n_rows, D, dtype=torch.float16, device="cuda")
    comp_v = torch.zeros_like(comp_k)
    state = torch.zeros(2 + 2 * D, dtype=torch.float32, device="cuda")
    rk, rv, wd = _dev(raw_k), _dev(raw_v), _dev(w)
    ds4a.ds4a_compress_append(rk[:p0], rv[:p0], wd, ratio, 0, state, comp_k, comp_v)
    torch.cuda.synchronize()
    qd, qid, kid = _dev(q), _dev(q_idx), _dev(kidx)
    out = torch.empty(S, H, D, dtype=torch.float16, device="cuda")
    if topk:
        sel = torch.full((topk,), -1, dtype=torch.int32, device="cuda")   # shared by every step
        sel_n = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = torch.zeros(ds4a.ds4a_indexer_workspace_bytes(1, kidx.shape[0], topk), dtype=torch.uint8,
                         device="cuda")
        sels = torch.empty(S, topk, dtype=torch.int32, device="cuda")
    for s in range(S):
        p = p0 + s
        n_vis = (p + 1) // ratio
        if fused and topk:   # the indexer query and the compressor update in one launch
            ds4a.ds4a_indexer_topk_compress(qid[s], kid, p, ratio, topk, sel, sel_n, ws, rk[p:p + 1], rv[p:p + 1],
                                            wd, state, comp_k, comp_v)
        elif not fused:
            if topk:
                ds4a.ds4a_indexer_topk(qid[s], kid, p, ratio, topk, sel, sel_n, ws)
            ds4a.ds4a_compress_append(rk[p:p + 1], rv[p:p + 1], wd, ratio, p, state, comp_k, comp_v)
        win = slice(p - W + 1, p + 1)
        if fused and not topk:   # the compressor update and the attention in one launch
            ds4a.ds4a_compress_attn_decode(rk[p:p + 1], rv[p:p + 1], wd, ratio, p, state, comp_k, comp_v, qd[s],
                                           rk[win], rv[win], scale, out[s])
        elif topk:
            ds4a.ds4a_attn_decode(qd[s], rk[win], rv[win], comp_k, comp_v, sel, topk, scale, out[s])
            sels[s].copy_(sel)   # a stream-ordered copy: the next indexer writes sel again
        else:
            ds4a.ds4a_attn_decode(qd[s], rk[win], rv[win], comp_k, comp_v, None, n_vis, scale, out[s])
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0

    ck, cv = oracle.compress_range(raw_k, raw_v, 0, w, ratio, 0, n_rows)
    check_out(comp_k.cpu().numpy(), ck, "pooled rows")
    check_out(comp_v.cpu().numpy(), cv, "pooled rows V")
    out_h = out.cpu().numpy()
    for s in range(S):
        p = p0 + s
        n_vis = (p + 1) // ratio
        if topk:
            idx, cnt = oracle.indexer(q_idx[s], kidx, p, ratio, topk)
            scores = oracle.index_scores(q_idx[s], kidx[:n_vis])
            check_sel(sels[s].cpu().numpy(), idx[0, : cnt[0]], scores, topk, f"sel step {s}")
            ref = oracle.decode_attend(q[s], p, W, raw_k, raw_v, 0, ck, cv, idx[0], topk, scale)
        else:
            ref = oracle.decode_attend(q[s], p, W, raw_k, raw_v, 0, ck, cv, None, n_vis, scale)
        check_out(out_h[s], ref, f"out step {s}")


def test_prefill_chunks_back_to_back():
    """Two 96-token chunks of a ratio-4 layer (H=64, D=128: the tensor-core kernels),
    the second issued right behind the first, sharing sel, the workspace and the state."""
    H, D, W, d_idx, topk, ratio, seed = 64, 128, 128, 128, 64, 4, 9
    P0, T = 400, 96
    n_tok = P0 + 2 * T
    raw_k = synth.normal_f16(seed, 2, synth.T_KRAW, (n_tok, D))
    raw_v = synth.normal_f16(seed, 2, synth.T_VRAW, (n_tok, D))
    w = synth.normal_f32(seed, 2, synth.T_W, (D,), 1.0 / math.sqrt(D))
    n_rows = n_tok // ratio
    kidx = synth.normal_f16(seed, 2, synth.T_KIDX, (n_rows, d_idx))
    q = synth.normal_f16(seed, 2, synth.T_Q, (2 * T, H, D))
    q_idx = synth.normal_f16(seed, 2, synth.T_QIDX, (2 * T, d_idx))
    scale = 1.0 / math.sqrt(D)

    rk, rv, wd = _dev(raw_k), _dev(raw_v), _dev(w)
    comp_k = torch.zeros(n_rows, D, dtype=torch.float16, device="cuda")
    comp_v = torch.zeros_like(comp_k)
    state = torch.zeros(2 + 2 * D, dtype=torch.float32, device="cuda")
    ds4a.ds4a_compress_append(rk[:P0], rv[:P0], wd, ratio, 0, state, comp_k, comp_v)
    torch.cuda.synchronize()
    qd, qid, kid = _dev(q), _dev(q_idx), _dev(kidx)
    sel = torch.full((T, topk), -1, dtype=torch.int32, device="cuda")
    sels = torch.empty(2, T, topk, dtype=torch.int32, device="cuda")
    ws = torch.zeros(ds4a.ds4a_indexer_workspace_bytes(T, n_rows, topk), dtype=torch.uint8, device="cuda")
    out = torch.empty(2 * T, H, D, dtype=torch.float16, device="cuda")
    for c in range(2):
        P = P0 + c * T
        n_prior = W - 1
        ds4a.ds4a_compress_append(rk[P:P + T], rv[P:P + T], wd, ratio, P, state, comp_k, comp_v)
        ds4a.ds4a_indexer_topk(qid[c * T:(c + 1) * T], kid, P, ratio, topk, sel, None, ws)
        ds4a.ds4a_attn_prefill(qd[c * T:(c + 1) * T], rk[P - n_prior:P + T], rv[P - n_prior:P + T], n_prior, W,
                               comp_k, comp_v, sel, P, ratio, scale, out[c * T:(c + 1) * T])
        sels[c].copy_(sel)
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0

    ck, cv = oracle.compress_range(raw_k, raw_v, 0, w, ratio, 0, n_rows)
    check_out(comp_k.cpu().numpy(), ck, "pooled rows")
    out_h, sels_h = out.cpu().numpy(), sels.cpu().numpy()
    for c in range(2):
        P = P0 + c * T
        idx, cnt = oracle.indexer(q_idx[c * T:(c + 1) * T], kidx, P, ratio, topk)
        for i in range(0, T, 7):
            n_vis = (P + i + 1) // ratio
            scores = oracle.index_scores(q_idx[c * T + i], kidx[:n_vis])
            check_sel(sels_h[c, i], idx[i, : cnt[i]], scores, topk, f"chunk {c} sel[{i}]")
            ref = oracle.decode_attend(q[c * T + i], P + i, W, raw_k, raw_v, 0, ck, cv, idx[i], topk, scale)
            check_out(out_h[c * T + i], ref, f"chunk {c} out[{i}]")
