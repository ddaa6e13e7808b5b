"""Decoding token after token through DecodeLayer.advance, across raw-window ring wraps.

Each advance appends the new token to the caller-held raw window ring (slot
p % W, overwriting the token that leaves the window), feeds it to the
compressor, runs the indexer and attention at the new position.  A run of S >= 2W
steps wraps the ring at least twice and crosses several block boundaries, so
that pooled rows completed during the run are attended (and, on a ratio-4
layer, ranked by the indexer) in later steps.  The steps are issued back to
back with no host synchronisation; every step's kept rows and output are then
compared with the oracle run on the token history up to that step.
("DS4 (DwarfStar 4)", Key Techniques, "KV attention compression" and "KV cache
with disk as first-class citizen": the 128-token raw sliding window and the
compressor fed one token at a time.)
"""
import math

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import synth
from compressed_sparse_mqa_gb300.layer import DecodeLayer
from parity import check_out, check_sel

pytestmark = pytest.mark.gpu


def _history(seed, H, D, W, ratio, d_idx, topk, p0, S):
    """Token history 0 .. p0 + S, indexer keys for every row it completes, and the
    queries of steps p0 .. p0 + S."""
    p_end = p0 + S
    raw_k = synth.normal_f16(seed, 7, synth.T_KRAW, (p_end + 1, D))
    raw_v = synth.normal_f16(seed, 7, synth.T_VRAW, (p_end + 1, D))
    n_rows = (p_end + 1) // ratio
    kidx = synth.normal_f16(seed, 7, synth.T_KIDX, (n_rows if topk else 0, d_idx))
    q = synth.normal_f16(seed, 7, synth.T_Q, (S + 1, H, D))
    q_idx = synth.normal_f16(seed, 7, synth.T_QIDX, (S + 1, d_idx) if topk else (S + 1, 0))
    w = synth.normal_f32(seed, 7, synth.T_W, (D,), 1.0 / math.sqrt(D))
    return raw_k, raw_v, kidx, q, q_idx, w


def _instance(p, H, D, W, ratio, d_idx, topk, raw_k, raw_v, kidx, q, q_idx, w):
    n_vis = (p + 1) // ratio
    return synth.DecodeInstance(H=H, D=D, window=W, ratio=ratio, d_idx=d_idx, topk=topk, p=p, pooled_history=True,
                                raw_pos0=0, raw_k=raw_k[: p + 1], raw_v=raw_v[: p + 1],
                                comp_k=np.zeros((0, D), np.float16), comp_v=np.zeros((0, D), np.float16),
                                kidx=kidx[:n_vis] if topk else kidx, q=q, q_idx=q_idx, w=w)


# (H, D, W, ratio, d_idx, topk, p0, S): S >= 2W steps each
CASES = [
    (8, 64, 32, 4, 32, 16, 200, 70),          # small ratio-4 layer with indexer
    (8, 64, 32, 128, 32, 0, 1000, 70),        # small ratio-128 layer (crosses the block ending at 1023)
    (64, 128, 128, 4, 128, 512, 4000, 260),   # model-sized ratio-4 layer: 1000 .. 1065 visible rows, top-512
    (64, 128, 128, 128, 128, 0, 1000, 300),   # model-sized ratio-128 layer: rows 7 .. 10 completed in the run
]


@pytest.mark.parametrize("H,D,W,ratio,d_idx,topk,p0,S", CASES)
def test_decode_advance_across_ring_wraps(H, D, W, ratio, d_idx, topk, p0, S):
    assert S >= 2 * W
    raw_k, raw_v, kidx, q, q_idx, w = _history(3, H, D, W, ratio, d_idx, topk, p0, S)
    inst0 = _instance(p0, H, D, W, ratio, d_idx, topk, raw_k, raw_v, kidx, q[0], q_idx[0], w)
    L = DecodeLayer(inst0, cap_extra=S // ratio + 2)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    rk, rv, qd, qid, kd = dev(raw_k), dev(raw_v), dev(q), dev(q_idx), dev(kidx)
    outs = torch.empty(S + 1, H, D, dtype=torch.float16, device="cuda")
    sels = torch.empty(S + 1, max(topk, 1), dtype=torch.int32, device="cuda")
    L.step()
    outs[0].copy_(L.out)
    if topk:
        sels[0].copy_(L.sel)
    for s in range(1, S + 1):
        p = p0 + s
        n_vis = (p + 1) // ratio
        completes = (p + 1) % ratio == 0
        L.advance(rk[p], rv[p], qd[s], qid[s] if topk else None,
                  kd[n_vis - 1] if (topk and completes) else None)
        outs[s].copy_(L.out)
        if topk:
            sels[s].copy_(L.sel)
    torch.cuda.synchronize()
    assert L.p == p0 + S
    from compressed_sparse_mqa_gb300 import ds4a
    assert ds4a.ds4a_last_device_error() == 0

    out_h, sel_h = outs.cpu().numpy(), sels.cpu().numpy()
    for s in range(S + 1):
        p = p0 + s
        inst = _instance(p, H, D, W, ratio, d_idx, topk, raw_k, raw_v, kidx, q[s], q_idx[s] if topk else q_idx[0], w)
        ref = oracle.decode_step(inst)
        if topk:
            scores = oracle.index_scores(q_idx[s], kidx[: ref["n_vis"]])
            check_sel(sel_h[s], ref["sel"], scores, topk, f"sel at p={p}")
        check_out(out_h[s], ref["out"], f"out at p={p}")
    # every row completed during the run was pooled by the GPU's online compressor
    n_end = (p0 + S + 1) // ratio
    ck, cv = oracle.compress_range(raw_k, raw_v, 0, w, ratio, 0, n_end)
    check_out(L.comp_k.cpu().numpy()[:n_end], ck, "pooled rows K")
    check_out(L.comp_v.cpu().numpy()[:n_end], cv, "pooled rows V")
    # the ring holds exactly the last W tokens, token t in slot t % W
    p_last = p0 + S
    ring_k = L.ring_k.cpu().numpy()
    for t in range(p_last - W + 1, p_last + 1):
        assert np.array_equal(ring_k[t % W], raw_k[t]), t


def test_restore_mid_block_continues_bit_for_bit():
    """A snapshot taken between two steps in the middle of a compressor block (both the
    ratio-4 and the ratio-128 block open), restored into freshly built layers, must
    continue exactly as the uninterrupted run: the same kept rows, outputs, pooled
    rows and compressor state, bit for bit.  ("DS4 (DwarfStar 4)", Key Techniques,
    "KV cache with disk as first-class citizen": snapshots carry the raw window rows
    and the compressor/indexer frontiers.)"""
    from compressed_sparse_mqa_gb300 import snapshot
    H, D, W, d_idx, p0, S1, S2 = 64, 128, 128, 128, 3000, 141, 150
    assert (p0 + S1 + 1) % 4 and (p0 + S1 + 1) % 128          # mid-block at the snapshot
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    specs = [(0, 0), (4, 512), (128, 0)]                       # window only, indexer layer, ratio 128
    hist = [_history(11 + i, H, D, W, r if r else 4, d_idx, k, p0, S1 + S2) for i, (r, k) in enumerate(specs)]

    def build():
        out = []
        for (r, k), (raw_k, raw_v, kidx, q, q_idx, w) in zip(specs, hist):
            if r == 0:
                inst = synth.DecodeInstance(H=H, D=D, window=W, ratio=0, d_idx=d_idx, topk=0, p=p0,
                                            pooled_history=False, raw_pos0=0, raw_k=raw_k[: p0 + 1],
                                            raw_v=raw_v[: p0 + 1], comp_k=np.zeros((0, D), np.float16),
                                            comp_v=np.zeros((0, D), np.float16), kidx=np.zeros((0, d_idx), np.float16),
                                            q=q[0], q_idx=np.zeros(0, np.float16), w=w)
            else:
                inst = _instance(p0, H, D, W, r, d_idx, k, raw_k, raw_v, kidx, q[0], q_idx[0] if k else q_idx[0], w)
            out.append(DecodeLayer(inst, cap_extra=(S1 + S2) // (r if r else 4) + 2))
        return out

    def run(layers, s_from, s_to, record):
        for s in range(s_from, s_to):
            p = p0 + s
            for L, (r, k), (raw_k, raw_v, kidx, q, q_idx, w), d in zip(layers, specs, hist, devs):
                n_vis = (p + 1) // r if r else 0
                completes = bool(r) and (p + 1) % r == 0
                L.advance(d[0][p], d[1][p], d[3][s], d[4][s] if k else None,
                          d[2][n_vis - 1] if (k and completes) else None)
                if record is not None:
                    record.append(L.out.clone())
                    if k:
                        record.append(L.sel.clone())

    devs = [(dev(a), dev(b), dev(c), dev(e), dev(f)) for a, b, c, e, f, _ in hist]
    A = build()
    for L in A:
        L.step()
    run(A, 1, S1 + 1, None)
    blob = snapshot.snapshot(A)
    rec_a = []
    run(A, S1 + 1, S1 + S2 + 1, rec_a)
    B = build()
    snapshot.restore(blob, B)
    assert [L.p for L in B] == [p0 + S1] * 3
    rec_b = []
    run(B, S1 + 1, S1 + S2 + 1, rec_b)
    torch.cuda.synchronize()
    assert len(rec_a) == len(rec_b) and rec_a
    for i, (x, y) in enumerate(zip(rec_a, rec_b)):
        assert torch.equal(x, y), f"record {i} differs after restore"
    for La, Lb in zip(A, B):
        assert torch.equal(La.state, Lb.state)
        if La.ratio:
            n = (La.p + 1) // La.ratio
            assert torch.equal(La.comp_k[:n], Lb.comp_k[:n]) and torch.equal(La.comp_v[:n], Lb.comp_v[:n])
    from compressed_sparse_mqa_gb300 import ds4a
    assert ds4a.ds4a_last_device_error() == 0
