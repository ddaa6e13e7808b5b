"""Batched decode: B independent sessions of one layer per launch.

("DwarfStar (ds4) Deep Dive", Step-by-Step Tutorial, "Start the Server": the
CUDA server serves 16 decode sessions with --batched-session 16.)  Each session
keeps its own position, raw window ring, compressed rows, indexer keys and
compressor state; the batched calls must give every session exactly what the
single-session calls give it -- the same kernels' arithmetic, so the same bits --
and each session must match the oracle.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import configs, ds4a, synth
from compressed_sparse_mqa_gb300.layer import BatchedDecodeLayer, DecodeLayer
from parity import check_out, check_sel

pytestmark = pytest.mark.gpu


def h(t):
    return t.detach().cpu().numpy()


def _sessions(layer, positions, H=64, D=128, W=128, d_idx=128, pooled_history=False):
    """One instance per session (its own cache and queries), all sharing the layer's
    compressor score weights."""
    ratio, topk = (0, 0) if layer < 2 else ((4, 512) if layer % 2 == 0 else (128, 0))
    insts = [synth.decode_instance(seed=100 + s, layer=layer, H=H, D=D, window=W, ratio=ratio, d_idx=d_idx, topk=topk,
                                   p=p, pooled_history=pooled_history, sigma_w=configs.SIGMA_W)
             for s, p in enumerate(positions)]
    return [dataclasses.replace(i, w=insts[0].w) for i in insts]


# positions: a plain step, a step that completes a block, an early position (k > visible
# rows, window not full), a different context length
@pytest.mark.parametrize("layer,positions", [(2, [32768, 32771, 20000, 5, 1023]),
                                             (3, [131072, 131071, 9000, 5]),
                                             (0, [5000, 70, 0])])
def test_batched_sessions_match_single_sessions_and_oracle(layer, positions):
    insts = _sessions(layer, positions)
    Bl = BatchedDecodeLayer(insts)
    singles = [DecodeLayer(i) for i in insts]
    Bl.step()
    outs = [L.step() for L in singles]
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    for s, (inst, L, out) in enumerate(zip(insts, singles, outs)):
        assert np.array_equal(h(Bl.out[s]), h(out)), f"session {s}: output differs from the single call"
        assert np.array_equal(h(Bl.state[s]), h(L.state)), f"session {s}: compressor state"
        if Bl.ratio:
            n = L.n_vis
            assert np.array_equal(h(Bl.comp_k[s, :n]), h(L.comp_k[:n])), f"session {s}: rows"
        if Bl.topk:
            assert np.array_equal(h(Bl.sel[s]), h(L.sel)), f"session {s}: kept rows"
            assert int(Bl.sel_n[s]) == int(L.sel_n)
        ref = oracle.decode_step(inst)
        if inst.topk:
            scores = oracle.index_scores(inst.q_idx, inst.kidx[: ref["n_vis"]])
            check_sel(h(Bl.sel[s]), ref["sel"], scores, inst.topk, f"session {s} sel")
        check_out(h(Bl.out[s]), ref["out"], f"session {s} out")


@pytest.mark.parametrize("layer", [2, 3])
def test_many_sessions_match_the_oracle(layer):
    """64 model-sized sessions in one call: more sessions than clusters of 16 can be
    resident at once, so the attention launch splits each session over a smaller
    cluster (a different split of its rows than the single-session call); every
    session's kept rows must still be exact and its output within the tolerance."""
    positions = [32768 + 37 * s for s in range(64)] if layer == 2 else [131071 + 129 * s for s in range(64)]
    insts = _sessions(layer, positions)
    Bl = BatchedDecodeLayer(insts)
    Bl.step()
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    out, sel = h(Bl.out), h(Bl.sel) if Bl.topk else None
    # the kept rows and the compressor's update are the single-session calls' bits
    # (the rows of a session are split differently across CTAs, the select is exact)
    for s in (0, 1, 31, 63):
        L = DecodeLayer(insts[s])
        L.step()
        torch.cuda.synchronize()
        assert np.array_equal(h(Bl.state[s]), h(L.state)), f"session {s}: compressor state"
        n = L.n_vis
        assert np.array_equal(h(Bl.comp_k[s, :n]), h(L.comp_k[:n])), f"session {s}: rows"
        if Bl.topk:
            assert np.array_equal(sel[s], h(L.sel)), f"session {s}: kept rows"
            assert int(Bl.sel_n[s]) == int(L.sel_n)
    for s, inst in enumerate(insts):
        ref = oracle.decode_step(inst)
        if inst.topk:
            scores = oracle.index_scores(inst.q_idx, inst.kidx[: ref["n_vis"]])
            check_sel(sel[s], ref["sel"], scores, inst.topk, f"session {s} sel")
        check_out(out[s], ref["out"], f"session {s} out")


@pytest.mark.parametrize("ratio,topk", [(4, 16), (128, 0)])
def test_batched_advance_across_ring_wraps(ratio, topk):
    """Three small sessions at different positions, 70 steps each (the ring of 32 wraps
    twice), every step of every session against the oracle."""
    H, D, W, d_idx, S = 8, 64, 32, 32, 70
    p0s = [200, 1001, 517] if ratio == 4 else [1000, 900, 1100]
    hist = []
    for s, p0 in enumerate(p0s):
        p_end = p0 + S
        rk = synth.normal_f16(40 + s, 1, synth.T_KRAW, (p_end + 1, D))
        rv = synth.normal_f16(40 + s, 1, synth.T_VRAW, (p_end + 1, D))
        ki = synth.normal_f16(40 + s, 1, synth.T_KIDX, ((p_end + 1) // ratio if topk else 0, d_idx))
        q = synth.normal_f16(40 + s, 1, synth.T_Q, (S + 1, H, D))
        qi = synth.normal_f16(40 + s, 1, synth.T_QIDX, (S + 1, d_idx))
        w = synth.normal_f32(7, 1, synth.T_W, (D,), 1.0 / math.sqrt(D))   # one layer: shared weights
        hist.append((rk, rv, ki, q, qi, w))

    def inst(s, p, step):
        rk, rv, ki, q, qi, w = hist[s]
        n_vis = (p + 1) // ratio
        return synth.DecodeInstance(H=H, D=D, window=W, ratio=ratio, d_idx=d_idx, topk=topk, p=p, pooled_history=True,
                                    raw_pos0=0, raw_k=rk[: p + 1], raw_v=rv[: p + 1],
                                    comp_k=np.zeros((0, D), np.float16), comp_v=np.zeros((0, D), np.float16),
                                    kidx=ki[:n_vis] if topk else ki, q=q[step], q_idx=qi[step] if topk else qi[0, :0],
                                    w=w)

    Bl = BatchedDecodeLayer([inst(s, p0, 0) for s, p0 in enumerate(p0s)], cap_extra=S // ratio + 2)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    outs = torch.empty(S + 1, len(p0s), H, D, dtype=torch.float16, device="cuda")
    sels = torch.empty(S + 1, len(p0s), max(topk, 1), dtype=torch.int32, device="cuda")
    Bl.step()
    outs[0].copy_(Bl.out)
    if topk:
        sels[0].copy_(Bl.sel)
    for step in range(1, S + 1):
        ps = [p0 + step for p0 in p0s]
        k = dev(np.stack([hist[s][0][p] for s, p in enumerate(ps)]))
        v = dev(np.stack([hist[s][1][p] for s, p in enumerate(ps)]))
        q = dev(np.stack([hist[s][3][step] for s in range(len(ps))]))
        qi = dev(np.stack([hist[s][4][step] for s in range(len(ps))])) if topk else None
        kr = None
        if topk:
            kr = dev(np.stack([hist[s][2][max(0, (p + 1) // ratio - 1)] for s, p in enumerate(ps)]))
        Bl.advance(k, v, q, qi, kr)
        outs[step].copy_(Bl.out)
        if topk:
            sels[step].copy_(Bl.sel)
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    out_h, sel_h = h(outs), h(sels)
    for step in range(S + 1):
        for s, p0 in enumerate(p0s):
            p = p0 + step
            ref = oracle.decode_step(inst(s, p, step))
            if topk:
                scores = oracle.index_scores(hist[s][4][step], hist[s][2][: ref["n_vis"]])
                check_sel(sel_h[step, s], ref["sel"], scores, topk, f"session {s} sel at p={p}")
            check_out(out_h[step, s], ref["out"], f"session {s} out at p={p}")


def test_batched_layer_refuses_sessions_with_different_weights():
    insts = _sessions(3, [1000, 1001], H=8, D=64, W=32, d_idx=32)
    other = dataclasses.replace(insts[1], w=insts[1].w + 1)
    with pytest.raises(ValueError, match="share"):
        BatchedDecodeLayer([insts[0], other])


def test_batched_capacity_overflow_is_recorded_not_written():
    """A session whose token would complete a row past its capacity: the compressor update
    is skipped and DS4A_ERR_CAPACITY recorded; the other sessions are unaffected."""
    insts = _sessions(3, [1000, 1001], H=8, D=64, W=32, d_idx=32, pooled_history=True)
    Bl = BatchedDecodeLayer(insts)          # capacity: 7 rows per session
    ref = Bl.clone()
    ref.step()
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    comp_before = h(Bl.comp_k).copy()
    Bl.pos[1] = 128 * Bl.cap + 127          # this token would complete row cap
    Bl.step()
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == ds4a.DS4A_ERR_CAPACITY
    assert np.array_equal(h(Bl.out[0]), h(ref.out[0]))
    assert np.array_equal(h(Bl.comp_k), comp_before)
    assert ds4a.ds4a_last_device_error() == 0
