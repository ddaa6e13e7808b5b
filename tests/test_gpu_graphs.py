"""The steps as the benchmark times them: captured in one CUDA graph over rotating
copies of the layer state, launched with programmatic dependent launch, replayed.
Every replayed step must give the bits of the same step issued eagerly on an
identical copy (same state, same order), so that the numbers the benchmark reports
are the numbers of the path the parity tests check against the oracle -- and the
first replayed step is also checked against the oracle directly.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import configs, ds4a, timing
from compressed_sparse_mqa_gb300.layer import BatchedDecodeLayer, DecodeLayer, PrefillLayer
from parity import check_out, check_sel

pytestmark = pytest.mark.gpu


def _replay_vs_eager(make, R, n_steps, outputs):
    """Capture n_steps steps over R copies (step t on copy t % R), replay once, and
    compare every copy's outputs with an eager run of the same sequence on fresh copies."""
    stream = torch.cuda.Stream()
    graph_copies = make(R)
    eager_copies = [c.clone() for c in graph_copies]
    with torch.cuda.stream(stream):   # one eager step each first, as the benchmark warms up
        for c, e in zip(graph_copies, eager_copies):
            c.step()
            e.step()
    torch.cuda.synchronize()
    g = timing.capture_graph(lambda t: graph_copies[t % R].step(), n_steps, stream)
    g.replay()
    with torch.cuda.stream(stream):
        for t in range(n_steps):
            eager_copies[t % R].step()
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    for c, e in zip(graph_copies, eager_copies):
        for name in outputs:
            assert torch.equal(getattr(c, name), getattr(e, name)), name
    return graph_copies


@pytest.mark.parametrize("params", [configs.C2, configs.C2_POOLED, configs.C3])
def test_decode_step_graph_replay(params):
    inst = configs.decode(params)
    names = ["out", "state"] + (["sel", "sel_n"] if inst.topk else [])
    copies = _replay_vs_eager(lambda R: [DecodeLayer(inst)] + [DecodeLayer(inst) for _ in range(R - 1)], 4, 8, names)
    # a freshly built copy stepped once inside a graph matches the oracle
    L = DecodeLayer(inst)
    stream = torch.cuda.Stream()
    g = timing.capture_graph(lambda t: L.step(), 1, stream)
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.decode_step(inst)
    if inst.topk and not L.pooled_keys:
        scores = oracle.index_scores(inst.q_idx, inst.kidx[: ref["n_vis"]])
        check_sel(L.sel.cpu().numpy(), ref["sel"], scores, inst.topk)
    if not L.pooled_keys:   # pooled keys: fp16 rounding of the keys, checked in their own tests
        check_out(L.out.cpu().numpy(), ref["out"])
    assert copies


def test_batched_step_graph_replay():
    import dataclasses
    insts = [configs.decode(dict(configs.C2, seed=s)) for s in range(16)]
    insts = [dataclasses.replace(i, w=insts[0].w) for i in insts]
    _replay_vs_eager(lambda R: [BatchedDecodeLayer(insts) for _ in range(R)], 2, 4, ["out", "sel", "sel_n", "state"])


def test_stack_graph_replay():
    """Two copies of the 43-layer stack at context 65536, one token each, in one graph."""
    class Stack:
        def __init__(self, layers):
            self.layers = layers

        def step(self):
            for L in self.layers:
                L.step()

        def clone(self):
            return Stack([L.clone() for L in self.layers])

    base = Stack([DecodeLayer(configs.decode(configs.c5_layer_params(l))) for l in range(43)])
    stream = torch.cuda.Stream()
    copies = [base, base.clone()]
    eager = [c.clone() for c in copies]
    g = timing.capture_graph(lambda t: copies[t % 2].step(), 2, stream)
    g.replay()
    with torch.cuda.stream(stream):
        for t in range(2):
            eager[t % 2].step()
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    for c, e in zip(copies, eager):
        for Lc, Le in zip(c.layers, e.layers):
            assert torch.equal(Lc.out, Le.out) and torch.equal(Lc.state, Le.state)
            if Lc.topk:
                assert torch.equal(Lc.sel, Le.sel)


def test_prefill_chunk_graph_replay():
    """The C4 chunk (compressor, indexer, attention) replayed from a graph over two
    copies gives the eager chunk's bits."""
    inst = configs.prefill(configs.C4)
    copies = [PrefillLayer(inst), PrefillLayer(inst)]
    eager = [PrefillLayer(inst), PrefillLayer(inst)]
    stream = torch.cuda.Stream()
    g = timing.capture_graph(lambda t: copies[t % 2].step(), 2, stream)
    g.replay()
    with torch.cuda.stream(stream):
        for t in range(2):
            eager[t % 2].step()
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    for c, e in zip(copies, eager):
        for name in ("out", "sel", "sel_n", "comp_k", "comp_v"):
            assert torch.equal(getattr(c, name), getattr(e, name)), name


def test_host_step_repeats_bit_for_bit():
    """The end-to-end call (host buffers in, output out) repeated at one position, as
    the benchmark's e2e loop does, gives the device step's bits every time."""
    inst = configs.decode(configs.C2)
    A, B = DecodeLayer(inst), DecodeLayer(inst)
    pin = lambda t: t.detach().cpu().pin_memory()
    out_h = torch.empty(A.H, A.D, dtype=torch.float16).pin_memory()
    run = B.bind_host(pin(B.ring_k[B.slot]), pin(B.ring_v[B.slot]), pin(B.q), pin(B.q_idx), out_h)
    for _ in range(4):
        A.step()
        run()
        assert torch.equal(out_h, A.out.cpu())
    assert ds4a.ds4a_last_device_error() == 0
    assert np.isfinite(out_h.float().numpy()).all()
