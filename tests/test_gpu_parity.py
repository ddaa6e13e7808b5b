"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Every test draws seeded synthetic inputs, runs the library's kernels on cuda:0
and compares with the oracle on the same inputs: outputs within max abs 2e-3 and
normwise rel 1e-2; kept indexer rows bit-exact up to near-ties (1e-6 relative of
the k-th score).  Every configuration, the full-size prefill chunk included, is
compared on every output.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import configs, ds4a, synth
from compressed_sparse_mqa_gb300.layer import DecodeLayer, PrefillLayer
from parity import check_out, check_sel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(ds4a_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    ds4a.ds4a_last_device_error()
    yield
    torch.cuda.synchronize()


def h(t):
    return t.detach().cpu().numpy()


def check_decode(inst, L=None):
    L = L or DecodeLayer(inst)
    out = L.step()
    torch.cuda.synchronize()
    ref = oracle.decode_step(inst)
    if inst.ratio and ref["comp_k"] is not None and ref["comp_k"].shape[0]:
        n = ref["comp_k"].shape[0]
        check_out(h(L.comp_k)[:n], ref["comp_k"], "comp_k")
        check_out(h(L.comp_v)[:n], ref["comp_v"], "comp_v")
    if inst.topk:
        scores = oracle.index_scores(inst.q_idx, inst.kidx[: ref["n_vis"]])
        check_sel(h(L.sel), ref["sel"], scores, inst.topk)
        assert int(L.sel_n.item()) == min(inst.topk, ref["n_vis"])
        assert (h(L.sel)[int(L.sel_n.item()):] == -1).all()
    check_out(h(out), ref["out"])
    assert ds4a.ds4a_last_device_error() == 0
    return L, ref


# ---- the five configurations ---------------------------------------------------------

def test_c1_tiny_even_layer_decode():
    inst = configs.decode(configs.C1)
    L, ref = check_decode(inst)
    assert ref["n_vis"] == 128 and len(ref["sel"]) == 16
    # the compressor produced all 128 rows from the raw tokens on the GPU
    assert np.abs(h(L.comp_k)).max() > 0


def test_c2_decode_ratio4_indexer():
    check_decode(configs.decode(configs.C2))


def test_c3_decode_ratio128_all_rows():
    check_decode(configs.decode(configs.C3))


def test_c3_decode_step_that_emits_a_row():
    inst = configs.decode(configs.C3_EMIT)
    L, ref = check_decode(inst)
    # row 1023 was pooled by this step from the 127 earlier tokens plus the current one
    check_out(h(L.comp_k)[1023], ref["comp_k"][1023], "row 1023 K")
    check_out(h(L.comp_v)[1023], ref["comp_v"][1023], "row 1023 V")


def test_c4_prefill_chunk_full():
    """The full-size prefill chunk checked on every query: all 2048 kept-row lists
    bit-exact (up to near-ties of the 512th score) and every output within tolerance.
    The oracle runs the whole chunk (about 20 GFLOP in double) in one call."""
    inst = configs.prefill(configs.C4)
    L = PrefillLayer(inst)
    L.step()
    torch.cuda.synchronize()
    P, T, r = inst.P, inst.T, inst.ratio
    ref = oracle.prefill_chunk(inst)
    # new pooled rows 7680 .. 8191
    check_out(h(L.comp_k)[P // r:], ref["new_k"], "new comp_k")
    check_out(h(L.comp_v)[P // r:], ref["new_v"], "new comp_v")
    sel_gpu, out_gpu = h(L.sel), h(L.out)
    assert np.array_equal(h(L.sel_n), ref["sel_n"])
    n_swapped = 0
    for i in range(T):
        n = int(ref["sel_n"][i])
        if np.array_equal(sel_gpu[i], ref["sel"][i]):
            continue
        n_vis = (P + i + 1) // r
        scores = oracle.index_scores(inst.q_idx[i], inst.kidx[:n_vis])
        n_swapped += check_sel(sel_gpu[i], ref["sel"][i, :n], scores, inst.topk, f"sel[{i}]")
    for i in range(T):
        check_out(out_gpu[i], ref["out"][i], f"out[{i}]")
    assert ds4a.ds4a_last_device_error() == 0


def test_c5_full_43_layer_stack():
    for layer in range(configs.C5_LAYERS):
        inst = configs.decode(configs.c5_layer_params(layer))
        check_decode(inst)


# ---- smaller prefill chunks, checked on every output ---------------------------------------

# (128, 0, 40000, ...): three compressed-row tiles without sel; (4, 1024, ...): a key list of
# 9 tiles, past the tensor-core kernel's 6, so the mma.sync kernel takes it
@pytest.mark.parametrize("ratio,topk,P,T,W", [(4, 16, 200, 96, 32), (4, 512, 2100, 130, 128),
                                              (128, 0, 300, 200, 128), (0, 0, 50, 77, 128),
                                              (4, 16, 0, 40, 32), (128, 0, 1000, 257, 64),
                                              (128, 0, 40000, 64, 128), (4, 1024, 8000, 64, 128)])
def test_prefill_small_full(ratio, topk, P, T, W):
    inst = synth.prefill_instance(seed=11, layer=ratio, H=64, D=128, window=W, ratio=ratio, d_idx=128,
                                  topk=topk, P=P, T=T, sigma_w=configs.SIGMA_W)
    L = PrefillLayer(inst)
    L.step()
    torch.cuda.synchronize()
    ref = oracle.prefill_chunk(inst)
    if ratio:
        n0 = P // ratio
        check_out(h(L.comp_k)[n0:], ref["new_k"], "new comp_k")
        check_out(h(L.comp_v)[n0:], ref["new_v"], "new comp_v")
    if topk:
        sel = h(L.sel)
        for i in range(T):
            n_vis = (P + i + 1) // ratio
            scores = oracle.index_scores(inst.q_idx[i], inst.kidx[:n_vis])
            check_sel(sel[i], ref["sel"][i, : ref["sel_n"][i]], scores, topk, f"sel[{i}]")
        assert np.array_equal(h(L.sel_n), ref["sel_n"])
    check_out(h(L.out), ref["out"])
    assert ds4a.ds4a_last_device_error() == 0


# ---- decode edge cases ------------------------------------------------------------------------

@pytest.mark.parametrize("p", [0, 2, 3, 17, 40, 131])
def test_decode_early_positions(p):
    # window not yet full, no or few compressed rows, k larger than the visible rows
    check_decode(synth.decode_instance(**dict(configs.C1, p=p)))


@pytest.mark.parametrize("H,D", [(8, 64), (64, 64), (8, 128), (24, 128), (64, 128)])
def test_decode_head_shapes(H, D):
    check_decode(synth.decode_instance(seed=5, layer=1, H=H, D=D, window=64, ratio=4, d_idx=64, topk=32,
                                       p=1000, sigma_w=0.1))


def test_decode_window_only_layer():
    check_decode(configs.decode(configs.c5_layer_params(0, context=5000)))


def test_decode_ratio128_block_boundaries():
    for p in [127, 128, 255, 383, 1000]:
        check_decode(synth.decode_instance(seed=2, layer=3, H=64, D=128, window=128, ratio=128, d_idx=128,
                                           topk=0, p=p, pooled_history=True, sigma_w=configs.SIGMA_W))


def test_attn_decode_skips_padding_and_flags_bad_rows():
    inst = configs.decode(dict(configs.C2, p=4000))
    L = DecodeLayer(inst)
    L.step()
    torch.cuda.synchronize()
    sel = h(L.sel).copy()
    n_comp = L.comp_k.shape[0]
    bad = sel.copy()
    bad[5] = -1
    bad[9] = n_comp + 7          # out of range: skipped and recorded
    bad_t = torch.from_numpy(bad).cuda()
    out = torch.empty_like(L.out)
    ds4a.ds4a_attn_decode(L.q, L.ring_k[: L.n_win], L.ring_v[: L.n_win], L.comp_k, L.comp_v, bad_t,
                          len(bad), L.scale, out)
    assert ds4a.ds4a_last_device_error() == ds4a.DS4A_ERR_DEVICE_INDEX
    assert ds4a.ds4a_last_device_error() == 0          # cleared by the read
    keep = bad.copy()
    keep[9] = -1
    ref = oracle.decode_attend(inst.q, inst.p, inst.window, inst.raw_k, inst.raw_v, inst.raw_pos0,
                               inst.comp_k, inst.comp_v, keep, len(keep), inst.scale)
    check_out(h(out), ref)


# ---- indexer edge cases --------------------------------------------------------------------------

def _indexer_gpu(q_idx, kidx, q_pos0, ratio, k):
    q = torch.from_numpy(np.ascontiguousarray(q_idx)).cuda()
    kk = torch.from_numpy(np.ascontiguousarray(kidx)).cuda()
    n_q = q.shape[0] if q.dim() == 2 else 1
    out = torch.full((n_q, k), -7, dtype=torch.int32, device="cuda")
    out_n = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    ws = torch.zeros(ds4a.ds4a_indexer_workspace_bytes(n_q, kk.shape[0], k), dtype=torch.uint8, device="cuda")
    ds4a.ds4a_indexer_topk(q, kk, q_pos0, ratio, k, out, out_n, ws)
    torch.cuda.synchronize()
    return h(out), h(out_n), ws


def test_indexer_ties_go_to_lower_index():
    rng = np.random.default_rng(3)
    base = rng.standard_normal((40, 16)).astype(np.float16)
    kidx = np.concatenate([base, base, base[:20]])          # every score appears 2-3 times
    q = rng.standard_normal(16).astype(np.float16)
    for k in [1, 7, 40, 63, 99]:
        out, n, _ = _indexer_gpu(q, kidx, 4 * 100, 4, k)
        ref = oracle.topk(oracle.index_scores(q, kidx), k)
        assert n[0] == len(ref)
        assert np.array_equal(out[0, : n[0]], ref), k


def test_indexer_large_row_counts_use_global_keys():
    rng = np.random.default_rng(4)
    for n_rows in [24577, 40000]:
        kidx = rng.standard_normal((n_rows, 128)).astype(np.float16)
        q = rng.standard_normal((1, 128)).astype(np.float16)
        out, n, ws = _indexer_gpu(q, kidx, 4 * n_rows + 3, 4, 512)
        scores = oracle.index_scores(q[0], kidx)
        check_sel(out[0], oracle.topk(scores, 512), scores, 512)
        # the decode ticket is back at zero for the next call
        assert int(ws[:4].view(torch.int32).item()) == 0
    # many queries with more visible rows than shared memory holds
    kidx = rng.standard_normal((30000, 64)).astype(np.float16)
    q = rng.standard_normal((3, 64)).astype(np.float16)
    out, n, _ = _indexer_gpu(q, kidx, 4 * 29990, 4, 100)
    for i in range(3):
        n_vis = min(30000, (4 * 29990 + i + 1) // 4)
        scores = oracle.index_scores(q[i], kidx[:n_vis])
        check_sel(out[i], oracle.topk(scores, 100), scores, 100, f"q{i}")


def test_indexer_k_exceeds_visible_rows():
    rng = np.random.default_rng(5)
    kidx = rng.standard_normal((500, 32)).astype(np.float16)
    q = rng.standard_normal((4, 32)).astype(np.float16)
    out, n, _ = _indexer_gpu(q, kidx, 397, 4, 512)      # 99 .. 100 rows visible
    for i in range(4):
        n_vis = (397 + i + 1) // 4
        assert n[i] == n_vis
        assert np.array_equal(out[i, :n_vis], np.arange(n_vis))
        assert (out[i, n_vis:] == -1).all()


def test_indexer_repeated_calls_reuse_workspace():
    inst = configs.decode(configs.C2)
    L = DecodeLayer(inst)
    L.step()
    first = h(L.sel).copy()
    for _ in range(5):
        L.step()
    torch.cuda.synchronize()
    assert np.array_equal(h(L.sel), first)


@pytest.mark.parametrize("p", [1, 3, 202, 203, 8191])
def test_indexer_topk_compress_matches_the_two_calls(p):
    """The one-launch indexer query + compressor update for position p gives the same
    bits as ds4a_indexer_topk followed by ds4a_compress_append: kept rows, count,
    running state and pooled rows (p = 3, 203, 8191 complete a block; p = 1 sees no row)."""
    ratio, topk, d_idx, D, seed = 4, 64, 64, 128, 11
    n_rows = (p + 1) // ratio
    kidx = torch.from_numpy(synth.normal_f16(seed, 3, synth.T_KIDX, (max(n_rows, 1), d_idx))).cuda()[:n_rows]
    q_idx = torch.from_numpy(synth.normal_f16(seed, 3, synth.T_QIDX, (d_idx,))).cuda()
    tok_k = torch.from_numpy(synth.normal_f16(seed, 3, synth.T_KRAW, (p + 1, D))).cuda()
    tok_v = torch.from_numpy(synth.normal_f16(seed, 3, synth.T_VRAW, (p + 1, D))).cuda()
    w = torch.from_numpy(synth.normal_f32(seed, 3, synth.T_W, (D,), 1.0 / np.sqrt(D))).cuda()
    comp_k = torch.zeros(n_rows + 1, D, dtype=torch.float16, device="cuda")
    comp_v = torch.zeros_like(comp_k)
    state = torch.zeros(2 + 2 * D, dtype=torch.float32, device="cuda")
    if p:
        ds4a.ds4a_compress_append(tok_k[:p], tok_v[:p], w, ratio, 0, state, comp_k, comp_v)
    nb = ds4a.ds4a_indexer_workspace_bytes(1, n_rows, topk)
    outs = []
    for fused in (False, True):
        ck, cv, st = comp_k.clone(), comp_v.clone(), state.clone()
        sel = torch.full((topk,), 7, dtype=torch.int32, device="cuda")
        sel_n = torch.full((1,), 7, dtype=torch.int32, device="cuda")
        ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        if fused:
            ds4a.ds4a_indexer_topk_compress(q_idx, kidx, p, ratio, topk, sel, sel_n, ws, tok_k[p:p + 1],
                                            tok_v[p:p + 1], w, st, ck, cv)
        else:
            ds4a.ds4a_indexer_topk(q_idx, kidx, p, ratio, topk, sel, sel_n, ws)
            ds4a.ds4a_compress_append(tok_k[p:p + 1], tok_v[p:p + 1], w, ratio, p, st, ck, cv)
        torch.cuda.synchronize()
        outs.append([h(x) for x in (sel, sel_n, st, ck, cv, ws)])
    for name, a, b in zip(["sel", "sel_n", "state", "comp_k", "comp_v", "workspace"], *outs):
        assert np.array_equal(a, b), name
    assert int(outs[1][1][0]) == min(topk, n_rows)
    assert not outs[1][5][:256].any()   # the ticket is back at zero for the next call
    assert ds4a.ds4a_last_device_error() == 0


@pytest.mark.parametrize("ratio,p,H,D", [(128, 254, 64, 128), (128, 255, 64, 128), (128, 256, 8, 64), (4, 7, 8, 64),
                                         (4, 1, 64, 128), (128, 131071, 64, 128)])
def test_compress_attn_decode_matches_the_two_calls(ratio, p, H, D):
    """The one-launch compressor update + attention over every visible row gives the
    same bits as ds4a_compress_append followed by ds4a_attn_decode (sel = NULL):
    output, running state and pooled rows (p + 1 = 256, 8, 131072 complete a block,
    whose row is then attended; p = 1 at ratio 4 sees no compressed row)."""
    W, seed = 128, 12
    n_vis = (p + 1) // ratio
    tok_k = torch.from_numpy(synth.normal_f16(seed, 4, synth.T_KRAW, (p + 1, D))).cuda()
    tok_v = torch.from_numpy(synth.normal_f16(seed, 4, synth.T_VRAW, (p + 1, D))).cuda()
    w = torch.from_numpy(synth.normal_f32(seed, 4, synth.T_W, (D,), 1.0 / np.sqrt(D))).cuda()
    q = torch.from_numpy(synth.normal_f16(seed, 4, synth.T_Q, (H, D))).cuda()
    win = slice(max(0, p - W + 1), p + 1)
    comp_k = torch.zeros(n_vis + 1, D, dtype=torch.float16, device="cuda")
    comp_v = torch.zeros_like(comp_k)
    state = torch.zeros(2 + 2 * D, dtype=torch.float32, device="cuda")
    if p:
        ds4a.ds4a_compress_append(tok_k[:p], tok_v[:p], w, ratio, 0, state, comp_k, comp_v)
    scale = 1.0 / np.sqrt(D)
    outs = []
    for fused in (False, True):
        ck, cv, st = comp_k.clone(), comp_v.clone(), state.clone()
        out = torch.full((H, D), 7, dtype=torch.float16, device="cuda")
        if fused:
            ds4a.ds4a_compress_attn_decode(tok_k[p:p + 1], tok_v[p:p + 1], w, ratio, p, st, ck, cv, q, tok_k[win],
                                           tok_v[win], scale, out)
        else:
            ds4a.ds4a_compress_append(tok_k[p:p + 1], tok_v[p:p + 1], w, ratio, p, st, ck, cv)
            ds4a.ds4a_attn_decode(q, tok_k[win], tok_v[win], ck, cv, None, n_vis, scale, out)
        torch.cuda.synchronize()
        outs.append([h(x) for x in (out, st, ck, cv)])
    for name, a, b in zip(["out", "state", "comp_k", "comp_v"], *outs):
        assert np.array_equal(a, b), name
    assert ds4a.ds4a_last_device_error() == 0


@pytest.mark.parametrize("layer", [0, 2, 3])   # window only, ratio 4 + indexer, ratio 128
def test_bound_step_matches_step(layer):
    """DecodeLayer.bind() marshals the step once; its launches give the same bits as step()."""
    inst = configs.decode(configs.c5_layer_params(layer))
    a = DecodeLayer(inst)
    b = a.clone()
    out_a = h(a.step())
    run = b.bind()
    out_b = h(run())
    torch.cuda.synchronize()
    assert np.array_equal(out_a, out_b)
    for name in ("state", "comp_k", "comp_v", "sel"):
        ta, tb = getattr(a, name, None), getattr(b, name, None)
        if ta is not None:
            assert np.array_equal(h(ta), h(tb)), name
    assert ds4a.ds4a_last_device_error() == 0


# ---- compressor: chunk-split invariance and online == blockwise ----------------------------------

@pytest.mark.parametrize("ratio", [4, 128])
def test_compressor_chunk_split_and_token_by_token(ratio):
    rng = np.random.default_rng(6)
    D, n = 128, 700
    k = rng.standard_normal((n, D)).astype(np.float16)
    v = rng.standard_normal((n, D)).astype(np.float16)
    w = (rng.standard_normal(D) * configs.SIGMA_W).astype(np.float32)
    ref_k, ref_v = oracle.compress_range(k, v, 0, w, ratio, 0, n // ratio)
    kt, vt, wt = (torch.from_numpy(x).cuda() for x in (k, v, w))

    def run(splits):
        ck = torch.zeros(n // ratio, D, dtype=torch.float16, device="cuda")
        cv = torch.zeros_like(ck)
        st = torch.zeros(2 + 2 * D, dtype=torch.float32, device="cuda")
        pos = 0
        for s in splits:
            ds4a.ds4a_compress_append(kt[pos:pos + s], vt[pos:pos + s], wt, ratio, pos, st, ck, cv)
            pos += s
        torch.cuda.synchronize()
        return h(ck), h(cv)

    whole = run([n])
    chunks = run([1, 130, 255, 314])
    tokens = run([1] * n)
    for got in (whole, chunks, tokens):
        check_out(got[0], ref_k, "rows K")
        check_out(got[1], ref_v, "rows V")
    np.testing.assert_allclose(chunks[0].astype(np.float32), whole[0].astype(np.float32), atol=2e-3)
    np.testing.assert_allclose(tokens[1].astype(np.float32), whole[1].astype(np.float32), atol=2e-3)


def test_indexer_many_queries_tensor_core_path_with_ties():
    """Many queries take the tensor-core scoring path.  Heavily duplicated key rows
    put thousands of exact ties at the k-th score, which overflows the exactly
    rescored band and exercises the exact fallback; ties must go to the lower index."""
    rng = np.random.default_rng(8)
    base = rng.standard_normal((4, 128)).astype(np.float16)
    kidx = np.repeat(base, 2048, axis=0)                   # 8192 rows, 4 distinct
    q = rng.standard_normal((64, 128)).astype(np.float16)
    out, n, _ = _indexer_gpu(q, kidx, 4 * 8192, 4, 512)
    for i in range(64):
        ref = oracle.topk(oracle.index_scores(q[i], kidx), 512)
        assert np.array_equal(out[i], ref), i
    # random keys, many queries, mixed visibility (the approximate bracket + exact band path)
    kidx = rng.standard_normal((3000, 64)).astype(np.float16)
    q = rng.standard_normal((200, 64)).astype(np.float16)
    out, n, _ = _indexer_gpu(q, kidx, 4 * 2900, 4, 300)
    for i in range(0, 200, 7):
        n_vis = min(3000, (4 * 2900 + i + 1) // 4)
        scores = oracle.index_scores(q[i], kidx[:n_vis])
        check_sel(out[i], oracle.topk(scores, 300), scores, 300, f"q{i}")
    assert ds4a.ds4a_last_device_error() == 0
