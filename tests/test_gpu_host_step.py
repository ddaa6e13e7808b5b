"""One decode step of one layer from host memory (ds4a_decode_layer_step).

The call copies the token's inputs from host buffers into the layer's device
arrays, runs the launches the device calls make, copies the output back and
waits.  Its results must be those of the device path (DecodeLayer.advance) bit
for bit, step after step across ring wraps and block completions, on every kind
of layer ("DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": the
window-only layers, the ratio-4 layers with the indexer, the ratio-128 layers),
and the last step must match the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import ds4a, synth
from compressed_sparse_mqa_gb300.layer import DecodeLayer
from parity import check_out, check_sel

pytestmark = pytest.mark.gpu


def _history(seed, H, D, ratio, d_idx, topk, p0, S, pooled):
    p_end = p0 + S
    rk = synth.normal_f16(seed, 9, synth.T_KRAW, (p_end + 1, D))
    rv = synth.normal_f16(seed, 9, synth.T_VRAW, (p_end + 1, D))
    n_rows = (p_end + 1) // ratio if ratio else 0
    ki = synth.normal_f16(seed, 9, synth.T_KIDX, (n_rows if topk else 0, d_idx))
    kt = synth.normal_f16(seed, 9, synth.T_KIDX_TOK, (p_end + 1, d_idx)) if pooled else None
    q = synth.normal_f16(seed, 9, synth.T_Q, (S + 1, H, D))
    qi = synth.normal_f16(seed, 9, synth.T_QIDX, (S + 1, d_idx))
    w = synth.normal_f32(seed, 9, synth.T_W, (D,), 1.0 / math.sqrt(D))
    return rk, rv, ki, kt, q, qi, w


def _instance(p, H, D, W, ratio, d_idx, topk, hist, step):
    rk, rv, ki, kt, q, qi, w = hist
    n_vis = (p + 1) // ratio if ratio else 0
    inst = synth.DecodeInstance(H=H, D=D, window=W, ratio=ratio, d_idx=d_idx, topk=topk, p=p, pooled_history=True,
                                raw_pos0=0, raw_k=rk[: p + 1], raw_v=rv[: p + 1],
                                comp_k=np.zeros((0, D), np.float16), comp_v=np.zeros((0, D), np.float16),
                                kidx=ki[:n_vis] if (topk and kt is None) else np.zeros((0, d_idx), np.float16),
                                q=q[step], q_idx=qi[step] if topk else np.zeros(0, np.float16), w=w,
                                kidx_tok=None if kt is None else kt[: p + 1])
    return inst


# (H, D, W, ratio, d_idx, topk, pooled, p0, S, pinned): page-locked buffers go through the
# input kernel and the direct output write, pageable ones through one copy per array
CASES = [
    (8, 64, 32, 0, 32, 0, False, 40, 70, True),              # window only
    (8, 64, 32, 128, 32, 0, False, 1000, 70, True),          # every row attended; completes row 7 at 1023
    (8, 64, 32, 4, 32, 16, False, 200, 70, True),            # indexer layer
    (8, 64, 32, 4, 32, 16, True, 200, 70, True),             # indexer layer pooling its keys
    (64, 128, 128, 4, 128, 512, False, 4000, 20, True),      # model-sized indexer layer
    (8, 64, 32, 4, 32, 16, False, 200, 30, False),           # indexer layer, pageable buffers
    (8, 64, 32, 128, 32, 0, False, 1000, 30, False),         # ratio-128 layer, pageable buffers
    (64, 128, 128, 128, 128, 0, False, 131060, 16, True),    # model-sized ratio-128 layer: 72 rows a CTA (one
                                                             # 80-row tile); completes row 1023 at 131071
]


@pytest.mark.parametrize("H,D,W,ratio,d_idx,topk,pooled,p0,S,pinned", CASES)
def test_host_step_matches_device_advance(H, D, W, ratio, d_idx, topk, pooled, p0, S, pinned):
    hist = _history(5, H, D, ratio, d_idx, topk, p0, S, pooled)
    rk, rv, ki, kt, q, qi, w = hist
    A = DecodeLayer(_instance(p0, H, D, W, ratio, d_idx, topk, hist, 0), cap_extra=S // max(ratio, 1) + 2)
    assert A.pooled_keys == pooled
    B = A.clone()
    A.step()
    B.step()
    host = lambda a: torch.from_numpy(np.ascontiguousarray(a)).clone()
    pin = (lambda a: host(a).pin_memory()) if pinned else host
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out_h = torch.empty(H, D, dtype=torch.float16)
    if pinned:
        out_h = out_h.pin_memory()
    for s in range(1, S + 1):
        p = p0 + s
        completes = bool(ratio) and (p + 1) % ratio == 0
        row = (p + 1) // ratio - 1 if ratio else -1
        krow = ki[row] if (topk and not pooled and completes) else None
        A.advance(dev(rk[p]), dev(rv[p]), dev(q[s]), dev(qi[s]) if topk else None,
                  dev(krow) if krow is not None else None, ki_tok=dev(kt[p]) if pooled else None)
        got = B.advance_host(pin(rk[p]), pin(rv[p]), pin(q[s]), pin(qi[s]) if topk else None,
                             pin(krow) if krow is not None else None, ki_tok=pin(kt[p]) if pooled else None,
                             out=out_h)
        assert got is out_h
        assert torch.equal(out_h, A.out.cpu()), f"output at p={p}"
        if not pinned:     # copied from the layer's out array
            assert torch.equal(B.out, A.out)
        if topk:
            assert torch.equal(A.sel, B.sel) and torch.equal(A.sel_n, B.sel_n), f"kept rows at p={p}"
    assert B.p == A.p == p0 + S and B.slot == A.slot and B.n_win == A.n_win and B.n_vis == A.n_vis
    assert torch.equal(A.ring_k, B.ring_k) and torch.equal(A.ring_v, B.ring_v) and torch.equal(A.state, B.state)
    if ratio:
        n = A.n_vis
        assert torch.equal(A.comp_k[:n], B.comp_k[:n]) and torch.equal(A.comp_v[:n], B.comp_v[:n])
    if topk:
        assert torch.equal(A.kidx[:A.n_vis], B.kidx[:B.n_vis])
    assert ds4a.ds4a_last_device_error() == 0
    # the last step against the oracle
    inst = _instance(p0 + S, H, D, W, ratio, d_idx, topk, hist, S)
    ref = oracle.decode_step(inst)
    if topk:
        keys = inst.kidx[: ref["n_vis"]]
        if pooled:       # the rows' keys pooled from their tokens' keys
            keys = oracle.compress_range_keys(rk, kt, 0, w, ratio, 0, ref["n_vis"])
        check_sel(B.sel.cpu().numpy(), ref["sel"], oracle.index_scores(qi[S], keys), topk, "sel")
    check_out(out_h.numpy(), ref["out"], "out")


def test_bound_host_step_repeats_the_device_step():
    """bind_host at a fixed position: each call gives the device step's output (the
    compressor state moves on each repeat on both sides alike)."""
    H, D, W, ratio, d_idx, topk, p0 = 64, 128, 128, 4, 128, 512, 32768
    hist = _history(8, H, D, ratio, d_idx, topk, p0, 0, False)
    A = DecodeLayer(_instance(p0, H, D, W, ratio, d_idx, topk, hist, 0))
    B = A.clone()
    pin = lambda t: t.detach().cpu().pin_memory()
    out_h = torch.empty(H, D, dtype=torch.float16).pin_memory()
    run = B.bind_host(pin(B.ring_k[B.slot]), pin(B.ring_v[B.slot]), pin(B.q), pin(B.q_idx), out_h)
    for _ in range(3):
        A.step()
        run()
        assert torch.equal(out_h, A.out.cpu())
        assert torch.equal(A.state, B.state) and torch.equal(A.sel, B.sel)
    # inputs already on the device and no read-back: the call only enqueues
    ds4a.ds4a_decode_layer_step(B.desc(), B.p)
    A.step()
    torch.cuda.synchronize()
    assert torch.equal(A.out, B.out)
    assert ds4a.ds4a_last_device_error() == 0
