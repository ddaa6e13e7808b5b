"""Host-side tests of the decode-state snapshot (no GPU needed).

The blob must carry every piece of per-layer state a later step reads -- the
position, the raw window ring, the compressor's running state, the compressed
rows and their indexer keys -- and nothing else; restoring it must reproduce
the state exactly, and a malformed or mismatching blob must be refused before
anything is written.  ("DS4 (DwarfStar 4)", Key Techniques, "KV cache with disk
as first-class citizen"; Design Decisions, "Innovation: disk KV as first-class
citizen".)
"""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

from compressed_sparse_mqa_gb300 import snapshot
from compressed_sparse_mqa_gb300.layer import layer_schedule


def _layer(layer, p, rng, H=8, D=64, W=32, d_idx=32, cap_extra=5, fill=True):
    ratio, topk = layer_schedule(layer)
    topk = 16 if topk else 0
    n = (p + 1) // ratio if ratio else 0
    cap = n + cap_extra
    f16 = lambda *s: torch.from_numpy(rng.standard_normal(s).astype(np.float16)) if fill else \
        torch.zeros(*s, dtype=torch.float16)
    L = SimpleNamespace(ratio=ratio, topk=topk, H=H, D=D, W=W, p=p, n_vis=n, slot=p % W, n_win=min(W, p + 1),
                        ring_k=f16(W, D), ring_v=f16(W, D),
                        state=torch.from_numpy(rng.standard_normal(2 + 2 * D).astype(np.float32)) if fill else
                        torch.zeros(2 + 2 * D),
                        comp_k=f16(cap, D) if ratio else None, comp_v=f16(cap, D) if ratio else None,
                        kidx=f16(cap, d_idx) if topk else None)
    return L


def _stack(p, rng, fill=True, layers=(0, 1, 2, 3, 4, 5)):
    return [_layer(l, p + l, rng, fill=fill) for l in layers]


def test_round_trip_restores_every_state_array():
    rng = np.random.default_rng(0)
    src = _stack(1000, rng)
    blob = snapshot.snapshot(src)
    dst = _stack(7, rng, fill=False)
    for d, s in zip(dst, src):      # same capacity as the source
        if s.ratio:
            d.comp_k = torch.zeros_like(s.comp_k)
            d.comp_v = torch.zeros_like(s.comp_v)
        if s.topk:
            d.kidx = torch.zeros_like(s.kidx)
        d.p = 7
    snapshot.restore(blob, dst)
    for s, d in zip(src, dst):
        assert d.p == s.p and d.n_vis == s.n_vis and d.slot == s.p % s.W and d.n_win == min(s.W, s.p + 1)
        assert torch.equal(d.ring_k, s.ring_k) and torch.equal(d.ring_v, s.ring_v)
        assert torch.equal(d.state, s.state)
        if s.ratio:
            n = (s.p + 1) // s.ratio
            assert torch.equal(d.comp_k[:n], s.comp_k[:n]) and torch.equal(d.comp_v[:n], s.comp_v[:n])
            assert not d.comp_k[n:].any()       # rows past the count are not state
        if s.topk:
            n = (s.p + 1) // s.ratio
            assert torch.equal(d.kidx[:n], s.kidx[:n])
    # the blob is deterministic and round-trips to itself
    assert snapshot.snapshot(dst) == blob


def test_blob_size_counts_exactly_the_state():
    rng = np.random.default_rng(1)
    src = _stack(500, rng)
    blob = snapshot.snapshot(src)
    expect = 16
    for L in src:
        n = (L.p + 1) // L.ratio if L.ratio else 0
        b = 64 + 2 * L.W * L.D * 2 + ((2 + 2 * L.D) * 4 + 15) // 16 * 16   # the state padded to 16 bytes
        if L.ratio:
            b += 2 * n * L.D * 2
        if L.topk:
            b += n * L.kidx.shape[1] * 2
        expect += b          # the row arrays here are 16-byte multiples already
    assert len(blob) == expect


def test_malformed_or_mismatching_blobs_are_refused_without_writing():
    rng = np.random.default_rng(2)
    src = _stack(300, rng)
    blob = snapshot.snapshot(src)
    dst = _stack(300, rng)
    before = [(L.ring_k.clone(), L.state.clone(), L.p) for L in dst]
    bad = [blob[:-20],                                    # truncated
           b"XXXXXXXX" + blob[8:],                        # magic
           blob[:8] + (2).to_bytes(4, "little") + blob[12:],   # version
           blob[:12] + (5).to_bytes(4, "little") + blob[16:]]  # layer count
    for b in bad:
        with pytest.raises(snapshot.SnapshotError):
            snapshot.restore(b, dst)
    with pytest.raises(snapshot.SnapshotError):           # schedule mismatch (layers swapped)
        snapshot.restore(blob, dst[::-1])
    small = _stack(300, rng, layers=(0, 1, 2, 3, 4, 5))
    small[2].comp_k = small[2].comp_k[:10]                # capacity below the row count
    with pytest.raises(snapshot.SnapshotError):
        snapshot.restore(blob, small)
    for L, (rk, st, p) in zip(dst, before):
        assert torch.equal(L.ring_k, rk) and torch.equal(L.state, st) and L.p == p


def test_save_frontier_aligns_to_chunks():
    # a cold save trims 32 tail tokens, then aligns down to a 2048-token boundary
    assert snapshot.save_frontier(25000) == 24576
    assert snapshot.save_frontier(24608) == 24576     # 24608 - 32 = 24576
    assert snapshot.save_frontier(24600) == 22528
    assert snapshot.save_frontier(24600 - 25) == 22528      # 24575 - 32 < 24576
    assert snapshot.save_frontier(2080) == 2048       # 2080 - 32 = 2048
    assert snapshot.save_frontier(2079) == 0          # 2047 is below the first boundary
    assert snapshot.save_frontier(4096, cold=False) == 4096
    assert snapshot.save_frontier(10) == 0
