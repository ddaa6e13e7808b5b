"""The compressor pooling per-token indexer keys (ds4a_compress_append_keys).

"DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": the compressor
keeps a rolling score/KV state and the ratio-4 layers rank the pooled rows with
a learned indexer.  In the reading these tests cover, a row's indexer key is
pooled from its tokens' indexer keys with the block's own softmax weights.

Checked against the oracle: the pooled keys (online token by token, in chunks
and blockwise), the pooled K/V rows (the same bits as ds4a_compress_append), and
decode steps and a prefill chunk whose indexer ranks the pooled keys.  The GPU
stores a pooled key in fp16 and the oracle keeps it in fp64, so kept rows may
differ only among rows whose scores lie within the fp16 rounding bound of the
k-th score; outputs are compared wherever the kept rows agree.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import ds4a, synth
from compressed_sparse_mqa_gb300.layer import DecodeLayer
from parity import check_out, check_sel_rounded_keys

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("ratio,D,DI", [(4, 128, 128), (128, 128, 64), (4, 64, 32)])
def test_pooled_keys_chunks_and_tokens(ratio, D, DI):
    n = 3 * 128 + 77
    k = synth.normal_f16(21, ratio, synth.T_KRAW, (n, D))
    v = synth.normal_f16(21, ratio, synth.T_VRAW, (n, D))
    ki = synth.normal_f16(21, ratio, synth.T_KIDX_TOK, (n, DI))
    w = synth.normal_f32(21, ratio, synth.T_W, (D,), 1.0 / math.sqrt(D))
    n_rows = n // ratio
    ref_ki = oracle.compress_range_keys(k, ki, 0, w, ratio, 0, n_rows)
    ref_k, ref_v = oracle.compress_range(k, v, 0, w, ratio, 0, n_rows)
    kt, vt, kit, wt = dev(k), dev(v), dev(ki), dev(w)

    def run(splits, keys=True):
        ck = torch.zeros(n_rows, D, dtype=torch.float16, device="cuda")
        cv, cki = torch.zeros_like(ck), torch.zeros(n_rows, DI, dtype=torch.float16, device="cuda")
        st = torch.zeros(2 + 2 * D + (DI if keys else 0), dtype=torch.float32, device="cuda")
        pos = 0
        for s in splits:
            if keys:
                ds4a.ds4a_compress_append_keys(kt[pos:pos + s], vt[pos:pos + s], kit[pos:pos + s], wt, ratio, pos, st,
                                               ck, cv, cki)
            else:
                ds4a.ds4a_compress_append(kt[pos:pos + s], vt[pos:pos + s], wt, ratio, pos, st, ck, cv)
            pos += s
        torch.cuda.synchronize()
        return ck.cpu().numpy(), cv.cpu().numpy(), cki.cpu().numpy(), st.cpu().numpy()

    plain = run([n], keys=False)
    for splits in ([n], [1, 130, 255, n - 386], [1] * n):
        ck, cv, cki, st = run(splits)
        check_out(cki, ref_ki, f"pooled keys {splits[:3]}")
        check_out(ck, ref_k, "rows K")
        check_out(cv, ref_v, "rows V")
        if len(splits) == 1:
            # the K/V rows and their state are the plain compressor's bits
            assert np.array_equal(ck, plain[0]) and np.array_equal(cv, plain[1])
            assert np.array_equal(st[: 2 + 2 * D], plain[3])
    assert ds4a.ds4a_last_device_error() == 0


# (H, D, W, d_idx, topk, p0, S)
@pytest.mark.parametrize("H,D,W,d_idx,topk,p0,S", [(8, 64, 32, 32, 16, 300, 70), (64, 128, 128, 128, 512, 4000, 40)])
def test_pooled_keys_decode_steps(H, D, W, d_idx, topk, p0, S):
    ratio, seed = 4, 23
    p_end = p0 + S
    inst_all = synth.decode_instance(seed=seed, layer=2, H=H, D=D, window=W, ratio=ratio, d_idx=d_idx, topk=topk,
                                     p=p_end, pooled_history=True, sigma_w=1.0 / math.sqrt(D), pooled_keys=True)
    raw_k, raw_v, ki = inst_all.raw_k, inst_all.raw_v, inst_all.kidx_tok   # positions 0 .. p_end
    q = synth.normal_f16(seed, 2, synth.T_Q, (S + 1, H, D))
    q_idx = synth.normal_f16(seed, 2, synth.T_QIDX, (S + 1, d_idx))

    def at(p, s):
        return synth.DecodeInstance(H=H, D=D, window=W, ratio=ratio, d_idx=d_idx, topk=topk, p=p,
                                    pooled_history=True, raw_pos0=0, raw_k=raw_k[: p + 1], raw_v=raw_v[: p + 1],
                                    comp_k=np.zeros((0, D), np.float16), comp_v=np.zeros((0, D), np.float16),
                                    kidx=np.zeros((0, d_idx), np.float16), q=q[s], q_idx=q_idx[s], w=inst_all.w,
                                    kidx_tok=ki[: p + 1])

    L = DecodeLayer(at(p0, 0), cap_extra=S // ratio + 2)
    assert L.pooled_keys
    rk, rv, kid, qd, qid = dev(raw_k), dev(raw_v), dev(ki), dev(q), dev(q_idx)
    outs = torch.empty(S + 1, H, D, dtype=torch.float16, device="cuda")
    sels = torch.empty(S + 1, topk, dtype=torch.int32, device="cuda")
    L.step()
    outs[0].copy_(L.out)
    sels[0].copy_(L.sel)
    for s in range(1, S + 1):
        p = p0 + s
        L.advance(rk[p], rv[p], qd[s], qid[s], ki_tok=kid[p])
        outs[s].copy_(L.out)
        sels[s].copy_(L.sel)
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    n_end = (p_end + 1) // ratio
    ref_keys = oracle.compress_range_keys(raw_k, ki, 0, inst_all.w, ratio, 0, n_end)
    check_out(L.kidx.cpu().numpy()[:n_end], ref_keys, "pooled keys")
    out_h, sel_h = outs.cpu().numpy(), sels.cpu().numpy()
    compared = 0
    for s in range(S + 1):
        p = p0 + s
        ref = oracle.decode_step(at(p, s))
        n_vis = (p + 1) // ratio
        diff = check_sel_rounded_keys(sel_h[s], ref["sel"], q_idx[s], ref_keys[:n_vis], f"sel at p={p}")
        if diff == 0:
            check_out(out_h[s], ref["out"], f"out at p={p}")
            compared += 1
    assert compared >= (S + 1) // 2


def test_pooled_keys_prefill_chunk():
    """A chunk pooled with its keys, then the many-query (tensor-core) indexer over the
    pooled keys -- issued right behind the compressor on the stream -- then attention."""
    H, D, W, d_idx, topk, ratio, seed = 64, 128, 128, 128, 64, 4, 27
    P, T = 600, 160
    n_tok = P + T
    k = synth.normal_f16(seed, 2, synth.T_KRAW, (n_tok, D))
    v = synth.normal_f16(seed, 2, synth.T_VRAW, (n_tok, D))
    ki = synth.normal_f16(seed, 2, synth.T_KIDX_TOK, (n_tok, d_idx))
    w = synth.normal_f32(seed, 2, synth.T_W, (D,), 1.0 / math.sqrt(D))
    q = synth.normal_f16(seed, 2, synth.T_Q, (T, H, D))
    q_idx = synth.normal_f16(seed, 2, synth.T_QIDX, (T, d_idx))
    n_rows = n_tok // ratio
    kt, vt, kit, wt = dev(k), dev(v), dev(ki), dev(w)
    ck = torch.zeros(n_rows, D, dtype=torch.float16, device="cuda")
    cv, cki = torch.zeros_like(ck), torch.zeros(n_rows, d_idx, dtype=torch.float16, device="cuda")
    st = torch.zeros(2 + 2 * D + d_idx, dtype=torch.float32, device="cuda")
    ds4a.ds4a_compress_append_keys(kt[:P], vt[:P], kit[:P], wt, ratio, 0, st, ck, cv, cki)
    torch.cuda.synchronize()
    sel = torch.full((T, topk), -1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(ds4a.ds4a_indexer_workspace_bytes(T, n_rows, topk), dtype=torch.uint8, device="cuda")
    out = torch.empty(T, H, D, dtype=torch.float16, device="cuda")
    n_prior = W - 1
    # back to back: the indexer ranks rows the compressor call just ahead of it writes
    ds4a.ds4a_compress_append_keys(kt[P:], vt[P:], kit[P:], wt, ratio, P, st, ck, cv, cki)
    ds4a.ds4a_indexer_topk(dev(q_idx), cki, P, ratio, topk, sel, None, ws)
    ds4a.ds4a_attn_prefill(dev(q), kt[P - n_prior:], vt[P - n_prior:], n_prior, W, ck, cv, sel, P, ratio,
                           1.0 / math.sqrt(D), out)
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    ref_keys = oracle.compress_range_keys(k, ki, 0, w, ratio, 0, n_rows)
    check_out(cki.cpu().numpy(), ref_keys, "pooled keys")
    ref_k, ref_v = oracle.compress_range(k, v, 0, w, ratio, 0, n_rows)
    idx, cnt = oracle.indexer(q_idx, ref_keys, P, ratio, topk)
    sel_h, out_h = sel.cpu().numpy(), out.cpu().numpy()
    compared = 0
    for i in range(T):
        n_vis = (P + i + 1) // ratio
        diff = check_sel_rounded_keys(sel_h[i], idx[i, : cnt[i]], q_idx[i], ref_keys[:n_vis], f"sel[{i}]")
        if diff == 0:
            ref = oracle.decode_attend(q[i], P + i, W, k, v, 0, ref_k, ref_v, idx[i], topk, 1.0 / math.sqrt(D))
            check_out(out_h[i], ref, f"out[{i}]")
            compared += 1
    assert compared >= T // 2


@pytest.mark.parametrize("ratio,p", [(4, 1), (4, 3), (4, 202), (4, 203), (4, 8191), (128, 1023), (128, 1100)])
def test_fused_pooled_step_matches_the_two_calls(ratio, p):
    """ds4a_indexer_topk_compress_keys gives the same bits as ds4a_compress_append_keys
    followed by ds4a_indexer_topk: kept rows, count, running state, pooled K/V rows and
    pooled indexer keys -- also when the token completes a row, which the launch's
    compressor CTA writes and scores (p = 3, 203, 8191, 1023) -- and leaves the
    workspace's completion count at zero."""
    topk, d_idx, D, seed = 64, 64, 128, 12
    n_done = p // ratio                 # rows complete before the token
    n_rows = (p + 1) // ratio + 2       # room for the row the token may complete
    ki_tok = dev(synth.normal_f16(seed, 5, synth.T_KIDX_TOK, (p + 1, d_idx)))
    q_idx = dev(synth.normal_f16(seed, 5, synth.T_QIDX, (d_idx,)))
    tok_k = dev(synth.normal_f16(seed, 5, synth.T_KRAW, (p + 1, D)))
    tok_v = dev(synth.normal_f16(seed, 5, synth.T_VRAW, (p + 1, D)))
    w = dev(synth.normal_f32(seed, 5, synth.T_W, (D,), 1.0 / math.sqrt(D)))
    comp_k = torch.zeros(n_rows, D, dtype=torch.float16, device="cuda")
    comp_v = torch.zeros_like(comp_k)
    kidx = torch.zeros(n_rows, d_idx, dtype=torch.float16, device="cuda")
    state = torch.zeros(2 + 2 * D + d_idx, dtype=torch.float32, device="cuda")
    if p:
        ds4a.ds4a_compress_append_keys(tok_k[:p], tok_v[:p], ki_tok[:p], w, ratio, 0, state, comp_k, comp_v, kidx)
    torch.cuda.synchronize()
    assert int((kidx[:n_done].abs().sum(dim=1) > 0).sum()) == n_done
    nb = ds4a.ds4a_indexer_workspace_bytes(1, n_rows, topk)
    outs = []
    for fused in (False, True):
        ck, cv, ki, st = comp_k.clone(), comp_v.clone(), kidx.clone(), state.clone()
        sel = torch.full((topk,), 7, dtype=torch.int32, device="cuda")
        sel_n = torch.full((1,), 7, dtype=torch.int32, device="cuda")
        ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        if fused:
            ds4a.ds4a_indexer_topk_compress_keys(q_idx, ki, p, ratio, topk, sel, sel_n, ws, tok_k[p:p + 1],
                                                 tok_v[p:p + 1], ki_tok[p:p + 1], w, st, ck, cv)
        else:
            ds4a.ds4a_compress_append_keys(tok_k[p:p + 1], tok_v[p:p + 1], ki_tok[p:p + 1], w, ratio, p, st, ck, cv,
                                           ki)
            ds4a.ds4a_indexer_topk(q_idx, ki, p, ratio, topk, sel, sel_n, ws)
        torch.cuda.synchronize()
        outs.append([x.cpu().numpy() for x in (sel, sel_n, st, ck, cv, ki, ws)])
    for name, a, b in zip(["sel", "sel_n", "state", "comp_k", "comp_v", "kidx", "workspace"], *outs):
        assert np.array_equal(a, b), name
    assert int(outs[1][1][0]) == min(topk, (p + 1) // ratio)
    assert not outs[1][6][:256].any()   # the completion count is back at zero for the next call
    assert ds4a.ds4a_last_device_error() == 0
