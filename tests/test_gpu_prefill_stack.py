"""One 2048-token prefill chunk through the full 43-layer schedule.

"DS4 (DwarfStar 4)", Architecture, "Whole-model graph execution" (prefill in
chunks of 2048 tokens) and Key Techniques, "KV attention compression" (layers
0-1 raw window only, even layers ratio 4 with the top-512 indexer, odd layers
ratio 128 attending every row).  The stack runs every layer back to back on one
stream; the test then checks, against the oracle, a layer of each kind: the
window-only layer 0 and the ratio-128 layer 3 on every query, the ratio-4 layer
2 on every kept-row list and on 256 queries spread over the chunk (the whole
ratio-4 chunk is checked on every output by the single-layer C4 test), and the
pooled rows every compressing layer appends.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import configs, ds4a
from compressed_sparse_mqa_gb300.layer import PrefillStack, layer_schedule
from parity import check_out, check_sel

pytestmark = pytest.mark.gpu


def test_prefill_stack_43_layers(ds4a_lib):
    torch.cuda.set_device(0)
    insts = configs.prefill_stack()
    assert len(insts) == 43
    stack = PrefillStack(insts)
    stack.step()
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    for l, (L, inst) in enumerate(zip(stack.layers, insts)):
        assert (L.ratio, L.topk) == layer_schedule(l)
        assert np.isfinite(L.out.float().cpu().numpy()).all(), l
    h = lambda t: t.detach().cpu().numpy()
    for l in (0, 3):                       # window only; ratio 128, every visible row
        inst, L = insts[l], stack.layers[l]
        ref = oracle.prefill_chunk(inst)
        if inst.ratio:
            n0 = inst.P // inst.ratio
            check_out(h(L.comp_k)[n0:], ref["new_k"], f"layer {l} new comp_k")
            check_out(h(L.comp_v)[n0:], ref["new_v"], f"layer {l} new comp_v")
        out = h(L.out)
        for i in range(inst.T):
            check_out(out[i], ref["out"][i], f"layer {l} out[{i}]")
    # ratio 4 + indexer: every kept-row list, 256 outputs spread over the chunk
    inst, L = insts[2], stack.layers[2]
    P, T, r = inst.P, inst.T, inst.ratio
    idx, cnt = oracle.indexer(inst.q_idx, inst.kidx, P, r, inst.topk)
    sel = h(L.sel)
    assert np.array_equal(h(L.sel_n), cnt)
    for i in range(T):
        if not np.array_equal(sel[i], idx[i]):
            scores = oracle.index_scores(inst.q_idx[i], inst.kidx[: (P + i + 1) // r])
            check_sel(sel[i], idx[i, : cnt[i]], scores, inst.topk, f"layer 2 sel[{i}]")
    nk, nv = oracle.compress_range(inst.raw_k, inst.raw_v, P - inst.n_prior, inst.w, r, P // r, (P + T) // r)
    check_out(h(L.comp_k)[P // r:], nk, "layer 2 new comp_k")
    comp_k = np.concatenate([inst.comp_k.astype(np.float64), nk])
    comp_v = np.concatenate([inst.comp_v.astype(np.float64), nv])
    out = h(L.out)
    for i in list(range(0, T, 8)) + [T - 1]:
        ref = oracle.decode_attend(inst.q[i], P + i, inst.window, inst.raw_k, inst.raw_v, P - inst.n_prior,
                                   comp_k, comp_v, idx[i], inst.topk, inst.scale)
        check_out(out[i], ref, f"layer 2 out[{i}]")
