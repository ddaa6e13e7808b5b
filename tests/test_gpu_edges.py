"""Edge cases of each step against the oracle: the smallest and largest sizes the
calls accept, the visible-row counts at which the decode select changes form,
empty inputs, and the degenerate compression ratios (1 and 1024).

("DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": the compressor
pools each block of `ratio` tokens, the indexer keeps the top-k rows, attention runs
one softmax over the window and the kept rows.)
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import configs, ds4a, synth
from compressed_sparse_mqa_gb300.layer import DecodeLayer, PrefillLayer
from parity import check_out, check_sel

pytestmark = pytest.mark.gpu


def h(t):
    return t.detach().cpu().numpy()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _indexer(q, kidx, q_pos0, ratio, k):
    qd, kd = dev(q), dev(kidx)
    n_q = qd.shape[0] if qd.dim() == 2 else 1
    out = torch.full((n_q, k), -7, dtype=torch.int32, device="cuda")
    out_n = torch.full((n_q,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(ds4a.ds4a_indexer_workspace_bytes(n_q, kd.shape[0], k), dtype=torch.uint8, device="cuda")
    ds4a.ds4a_indexer_topk(qd, kd, q_pos0, ratio, k, out, out_n, ws)
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    return h(out), h(out_n)


# one query: the select holds 8, 16 or 32 keys a thread up to 4096, 8192, 16384 visible
# rows and re-reads its keys from memory beyond; d_idx from 8 to 256, k up to 2048
@pytest.mark.parametrize("n_rows,d_idx,k", [(1, 8, 1), (4096, 128, 512), (4097, 24, 512), (8192, 256, 512),
                                            (8193, 128, 2048), (16384, 64, 512), (16385, 128, 512),
                                            (50000, 128, 2048)])
def test_indexer_one_query_sizes(n_rows, d_idx, k):
    rng = np.random.default_rng(n_rows + d_idx)
    kidx = rng.standard_normal((n_rows, d_idx)).astype(np.float16)
    q = rng.standard_normal((1, d_idx)).astype(np.float16)
    out, n = _indexer(q, kidx, 4 * n_rows + 3, 4, k)
    scores = oracle.index_scores(q[0], kidx)
    ref = oracle.topk(scores, k)
    assert n[0] == min(k, n_rows)
    check_sel(out[0], ref, scores, k)
    assert (out[0, n[0]:] == -1).all()


def test_indexer_no_visible_rows():
    """Early positions: no compressed row is complete yet -- every slot is -1 and the
    count 0, for one query and for many."""
    rng = np.random.default_rng(1)
    kidx = rng.standard_normal((64, 32)).astype(np.float16)
    for q_pos0, n_q in [(0, 1), (2, 1), (0, 64)]:   # at most k = 16 rows visible to any query
        q = rng.standard_normal((n_q, 32)).astype(np.float16)
        out, n = _indexer(q, kidx, q_pos0, 4, 16)
        for i in range(n_q):
            n_vis = (q_pos0 + i + 1) // 4
            assert n[i] == min(16, n_vis)
            assert np.array_equal(out[i, :n[i]], np.arange(n[i]))
            assert (out[i, n[i]:] == -1).all()


# many queries: the tensor-core scoring path (d_idx 64 / 128, up to 8192 rows) and the
# per-query kernel beyond it, k up to 2048
@pytest.mark.parametrize("n_q,n_rows,d_idx,k", [(64, 8192, 128, 2048), (65, 8193, 128, 512), (100, 3000, 32, 700)])
def test_indexer_many_query_sizes(n_q, n_rows, d_idx, k):
    rng = np.random.default_rng(n_q * n_rows)
    kidx = rng.standard_normal((n_rows, d_idx)).astype(np.float16)
    q = rng.standard_normal((n_q, d_idx)).astype(np.float16)
    q_pos0 = 4 * (n_rows - n_q // 2)           # the last queries see every row, the first ones fewer
    out, n = _indexer(q, kidx, q_pos0, 4, k)
    for i in list(range(0, n_q, 9)) + [n_q - 1]:
        n_vis = min(n_rows, (q_pos0 + i + 1) // 4)
        scores = oracle.index_scores(q[i], kidx[:n_vis])
        assert n[i] == min(k, n_vis)
        check_sel(out[i], oracle.topk(scores, k), scores, k, f"q{i}")


@pytest.mark.parametrize("ratio,D,n", [(1, 64, 300), (1024, 128, 2600), (3, 256, 400)])
def test_compressor_degenerate_ratios(ratio, D, n):
    """Ratio 1 (every token is its own row: the softmax over one token is 1, so the row
    is the token), the largest ratio 1024, and the largest head_dim 256, as one chunk
    and token by token."""
    rng = np.random.default_rng(ratio)
    k = rng.standard_normal((n, D)).astype(np.float16)
    v = rng.standard_normal((n, D)).astype(np.float16)
    w = (rng.standard_normal(D) * configs.SIGMA_W).astype(np.float32)
    rows = n // ratio
    ref_k, ref_v = oracle.compress_range(k, v, 0, w, ratio, 0, rows)
    kt, vt, wt = dev(k), dev(v), dev(w)
    for splits in ([n], [1] * n if n <= 400 else [1, 1023, 1, 1575]):
        ck = torch.zeros(max(rows, 1), D, dtype=torch.float16, device="cuda")
        cv = torch.zeros_like(ck)
        st = torch.zeros(2 + 2 * D, dtype=torch.float32, device="cuda")
        pos = 0
        for s in splits:
            ds4a.ds4a_compress_append(kt[pos:pos + s], vt[pos:pos + s], wt, ratio, pos, st, ck, cv)
            pos += s
        torch.cuda.synchronize()
        check_out(h(ck)[:rows], ref_k, f"rows K ({len(splits)} calls)")
        check_out(h(cv)[:rows], ref_v, f"rows V ({len(splits)} calls)")
    if ratio == 1:
        assert np.array_equal(h(ck)[:rows], k) and np.array_equal(h(cv)[:rows], v)
    assert ds4a.ds4a_last_device_error() == 0


@pytest.mark.parametrize("ratio,topk,window,p", [(1, 0, 128, 300), (4, 2048, 128, 40000), (4, 512, 4096, 20000),
                                                 (128, 0, 4096, 9000), (0, 0, 4096, 6000), (4, 512, 1, 5000),
                                                 (128, 0, 128, 114815), (128, 0, 128, 147500)])
def test_decode_extreme_shapes(ratio, topk, window, p):
    """A decode step with ratio 1 (every token a row), the largest k (2048), the
    largest window (4096 rows: up to 288 rows a CTA) and a one-row window; and a
    ratio-128 layer whose CTAs attend 65 rows each (a step that completes a row) and
    80 rows each, the bounds of the fused launch's one-tile form."""
    inst = synth.decode_instance(seed=21, layer=2, H=64, D=128, window=window, ratio=ratio, d_idx=128, topk=topk,
                                 p=p, sigma_w=configs.SIGMA_W)
    L = DecodeLayer(inst)
    out = L.step()
    torch.cuda.synchronize()
    ref = oracle.decode_step(inst)
    if topk:
        scores = oracle.index_scores(inst.q_idx, inst.kidx[: ref["n_vis"]])
        check_sel(h(L.sel), ref["sel"], scores, topk)
    check_out(h(out), ref["out"])
    assert ds4a.ds4a_last_device_error() == 0


@pytest.mark.parametrize("ratio,topk,P,T,W", [(4, 16, 300, 1, 32), (4, 512, 5000, 33, 1), (128, 0, 9000, 40, 4096),
                                              (0, 0, 5000, 20, 4096), (4, 2048, 12000, 64, 128)])
def test_prefill_extreme_shapes(ratio, topk, P, T, W):
    """A one-query chunk, a one-row window, the largest window (the kernel without the
    tensor-core key limit) and the largest k."""
    inst = synth.prefill_instance(seed=23, layer=2, H=64, D=128, window=W, ratio=ratio, d_idx=128, topk=topk, P=P,
                                  T=T, sigma_w=configs.SIGMA_W)
    L = PrefillLayer(inst)
    L.step()
    torch.cuda.synchronize()
    ref = oracle.prefill_chunk(inst)
    if ratio:
        n0 = P // ratio
        check_out(h(L.comp_k)[n0:], ref["new_k"], "new comp_k")
    if topk:
        sel = h(L.sel)
        for i in range(T):
            n_vis = (P + i + 1) // ratio
            scores = oracle.index_scores(inst.q_idx[i], inst.kidx[:n_vis])
            check_sel(sel[i], ref["sel"][i, : ref["sel_n"][i]], scores, topk, f"sel[{i}]")
    check_out(h(L.out), ref["out"])
    assert ds4a.ds4a_last_device_error() == 0
