"""Pins of the fp64 CPU oracle against facts that do not come from the oracle.

Each test checks one function of the oracle against a closed form, an
invariant the method must satisfy, brute force on a tiny input, or a library
routine that the special case reduces to (torch softmax / scaled-dot-product
attention in float64, numpy lexicographic sort).  Sources: "DS4 (DwarfStar 4)",
Key Techniques, "KV attention compression" (schedule, pooled rows, top-512
indexer) and Architecture (64 heads, one KV head, 128-token window).
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_mqa_gb300 import synth

rng = np.random.default_rng(1234)


def f16(shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


# ---- layer schedule and row counts -----------------------------------------

def test_layer_schedule_matches_pages():
    # layers 0-1 raw window only; even from 2: ratio 4 + top-512; odd: ratio 128, no indexer
    for layer in range(43):
        r, k = oracle.layer_ratio(layer), oracle.layer_topk(layer)
        if layer < 2:
            assert (r, k) == (0, 0)
        elif layer % 2 == 0:
            assert (r, k) == (4, 512)
        else:
            assert (r, k) == (128, 0)


@pytest.mark.parametrize("p,r,want", [(511, 4, 128), (512, 4, 128), (32768, 4, 8192),
                                      (131072, 128, 1024), (131071, 128, 1024), (131070, 128, 1023),
                                      (65536, 4, 16384), (65536, 128, 512), (30720, 4, 7680),
                                      (32767, 4, 8192), (0, 4, 0), (3, 4, 1), (5, 0, 0)])
def test_rows_visible_is_floor_prefix_over_ratio(p, r, want):
    assert oracle.rows_visible(p, r) == want
    if r:
        assert want == (p + 1) // r


# ---- compressor -------------------------------------------------------------

def test_ratio_one_pooling_is_identity():
    k, v, w = f16((37, 16)), f16((37, 16)), rng.standard_normal(16)
    ok, ov = oracle.compress_range(k, v, 0, w, 1, 0, 37)
    assert np.array_equal(ok, k.astype(np.float64))
    assert np.array_equal(ov, v.astype(np.float64))


@pytest.mark.parametrize("r", [4, 128])
def test_zero_score_weights_give_block_mean(r):
    n = 3 * r
    k, v = f16((n, 32)), f16((n, 32))
    ok, ov = oracle.compress_range(k, v, 0, np.zeros(32), r, 0, 3)
    # fp16 sums are exact in double, and 1/r is a power of two: exact equality
    assert np.array_equal(ok, k.astype(np.float64).reshape(3, r, 32).mean(axis=1))
    assert np.array_equal(ov, v.astype(np.float64).reshape(3, r, 32).mean(axis=1))


def test_constant_score_shift_cancels():
    r, D, d0 = 4, 16, 5
    k, v, w = f16((2 * r, D)), f16((2 * r, D)), rng.standard_normal(D)
    k[:, d0] = 0
    k2 = k.copy()
    k2[:r, d0] = 3.0     # constant inside block 0
    k2[r:, d0] = -2.5    # another constant inside block 1
    a_k, a_v = oracle.compress_range(k, v, 0, w, r, 0, 2)
    b_k, b_v = oracle.compress_range(k2, v, 0, w, r, 0, 2)
    np.testing.assert_allclose(b_v, a_v, rtol=0, atol=1e-12)
    keep = [d for d in range(D) if d != d0]
    np.testing.assert_allclose(b_k[:, keep], a_k[:, keep], rtol=0, atol=1e-12)
    np.testing.assert_allclose(b_k[:, d0], [3.0, -2.5], rtol=0, atol=1e-12)


def test_two_token_block_closed_form():
    # s = (0, 1): weights (1 - sigma(1), sigma(1)) with sigma(x) = 1/(1+e^-x)
    k = np.array([[0.0, 2.0], [1.0, -4.0]])
    v = np.array([[1.0, 0.5], [3.0, -1.0]])
    ok, ov = oracle.pool_block(k, v, np.array([1.0, 0.0]))
    a1 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(ok, (1 - a1) * k[0] + a1 * k[1], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(ov, (1 - a1) * v[0] + a1 * v[1], rtol=1e-15, atol=1e-15)


def test_pooling_equals_library_softmax_weighted_sum():
    r, D = 4, 16
    k, v = f16((5 * r, D)), f16((5 * r, D))
    w = rng.standard_normal(D)
    ok, ov = oracle.compress_range(k, v, 0, w, r, 0, 5)
    K = torch.tensor(k.astype(np.float64)).view(5, r, D)
    V = torch.tensor(v.astype(np.float64)).view(5, r, D)
    a = torch.softmax(K @ torch.tensor(w), dim=1)          # [5, r]
    np.testing.assert_allclose(ok, (a[..., None] * K).sum(1).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(ov, (a[..., None] * V).sum(1).numpy(), rtol=0, atol=1e-12)


def test_compress_range_offsets_and_bounds():
    r, D = 4, 8
    k, v, w = f16((40, D)), f16((40, D)), rng.standard_normal(D)
    full_k, full_v = oracle.compress_range(k, v, 0, w, r, 0, 10)
    # raw rows starting at position 12 reproduce blocks 3..9
    part_k, part_v = oracle.compress_range(k[12:], v[12:], 12, w, r, 3, 10)
    assert np.array_equal(part_k, full_k[3:])
    assert np.array_equal(part_v, full_v[3:])
    with pytest.raises(ValueError):
        oracle.compress_range(k[13:], v[13:], 13, w, r, 3, 10)   # block 3 starts at 12


# ---- pooled indexer keys (the compressor pooling per-token indexer keys) -------

def test_pooled_keys_ratio_one_is_identity():
    k, ki, w = f16((21, 16)), f16((21, 24)), rng.standard_normal(16)
    assert np.array_equal(oracle.compress_range_keys(k, ki, 0, w, 1, 0, 21), ki.astype(np.float64))


@pytest.mark.parametrize("r", [4, 128])
def test_pooled_keys_zero_weights_give_block_mean(r):
    k, ki = f16((2 * r, 16)), f16((2 * r, 40))
    got = oracle.compress_range_keys(k, ki, 0, np.zeros(16), r, 0, 2)
    assert np.array_equal(got, ki.astype(np.float64).reshape(2, r, 40).mean(axis=1))


def test_pooled_keys_two_token_closed_form():
    k = np.array([[0.0, 2.0], [1.0, -4.0]])
    ki = np.array([[5.0, -1.0, 0.25], [1.0, 3.0, -0.5]])
    got = oracle.pool_block_keys(k, ki, np.array([1.0, 0.0]))
    a1 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(got, (1 - a1) * ki[0] + a1 * ki[1], rtol=1e-15, atol=1e-15)


def test_pooled_keys_use_the_library_softmax_of_the_k_scores():
    # the weights come from w . k_t, not from the indexer keys: a library softmax of the
    # K scores applied to the indexer keys
    r, D, DI = 4, 16, 8
    k, ki, w = f16((6 * r, D)), f16((6 * r, DI)), rng.standard_normal(D)
    got = oracle.compress_range_keys(k, ki, 0, w, r, 0, 6)
    K = torch.tensor(k.astype(np.float64)).view(6, r, D)
    KI = torch.tensor(ki.astype(np.float64)).view(6, r, DI)
    a = torch.softmax(K @ torch.tensor(w), dim=1)
    np.testing.assert_allclose(got, (a[..., None] * KI).sum(1).numpy(), rtol=0, atol=1e-12)


def test_pooled_keys_offsets_and_bounds():
    r, D, DI = 4, 8, 16
    k, ki, w = f16((40, D)), f16((40, DI)), rng.standard_normal(D)
    full = oracle.compress_range_keys(k, ki, 0, w, r, 0, 10)
    assert np.array_equal(oracle.compress_range_keys(k[12:], ki[12:], 12, w, r, 3, 10), full[3:])
    with pytest.raises(ValueError):
        oracle.compress_range_keys(k[13:], ki[13:], 13, w, r, 3, 10)


# ---- indexer ------------------------------------------------------------------

def test_index_scores_on_orthonormal_keys():
    d = 8
    q = rng.standard_normal(d)
    s = oracle.index_scores(q, np.eye(d))
    np.testing.assert_array_equal(s, q)
    s2 = oracle.index_scores(q, -2.0 * np.eye(d)[::-1])
    np.testing.assert_array_equal(s2, -2.0 * q[::-1])


@pytest.mark.parametrize("n", [1, 5, 9, 12])
def test_topk_equals_subset_brute_force(n):
    for trial in range(5):
        s = rng.permutation(n).astype(np.float64) + rng.uniform(0, 0.5, n)   # distinct in fp32
        for k in range(1, n + 1):
            best = max(itertools.combinations(range(n), k), key=lambda c: sum(s[list(c)]))
            assert list(oracle.topk(s, k)) == sorted(best)


def test_topk_equals_lexicographic_sort_with_ties():
    for trial in range(20):
        n = int(rng.integers(1, 300))
        s = rng.integers(-5, 6, n).astype(np.float64)   # many exact ties
        k = int(rng.integers(1, 40))
        order = np.lexsort((np.arange(n), -s))           # score desc, then index asc
        assert list(oracle.topk(s, k)) == sorted(order[: min(k, n)].tolist())


def test_topk_ranks_in_binary32():
    # 1 + 1e-12 and 1 round to the same float: the tie goes to the lower index
    s = np.array([1.0, 1.0 + 1e-12, 0.5])
    assert list(oracle.topk(s, 1)) == [0]
    assert list(oracle.topk(s[::-1].copy(), 1)) == [1]


def test_topk_k_larger_than_rows():
    assert list(oracle.topk(np.array([3.0, -1.0, 2.0]), 16)) == [0, 1, 2]
    assert list(oracle.topk(np.zeros(0), 16)) == []


def test_indexer_respects_visibility_and_pads():
    d, n, r, k = 4, 40, 4, 6
    kidx = f16((n, d))
    q = (np.abs(f16((5, d))) + 0.25).astype(np.float16)
    # rows 5.. are never visible to positions 18..22 (ratio 4); give them the
    # largest scores so that ignoring visibility would pick them
    kidx[5:] = 50.0
    idx, cnt = oracle.indexer(q, kidx, q_pos0=18, ratio=r, k=k)
    for i in range(5):
        n_vis = (18 + i + 1) // r
        assert cnt[i] == min(k, n_vis)
        assert (idx[i, : cnt[i]] < n_vis).all()
        assert (idx[i, cnt[i]:] == -1).all()
        s = oracle.index_scores(q[i], kidx[:n_vis])
        assert list(idx[i, : cnt[i]]) == list(oracle.topk(s, k))
    idx0, cnt0 = oracle.indexer(q[:1], kidx, q_pos0=2, ratio=r, k=k)   # nothing visible yet
    assert cnt0[0] == 0 and (idx0 == -1).all()


# ---- attention -----------------------------------------------------------------

def sdpa64(q, K, V, scale):
    """Library multi-query attention in float64: q [H, D], K/V [n, D] shared by all heads."""
    qt = torch.tensor(np.asarray(q, dtype=np.float64))[None, :, None, :]        # [1, H, 1, D]
    H = qt.shape[1]
    Kt = torch.tensor(np.asarray(K, dtype=np.float64))[None, None].expand(1, H, -1, -1)
    Vt = torch.tensor(np.asarray(V, dtype=np.float64))[None, None].expand(1, H, -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    return o[0, :, 0, :].numpy()


def test_attend_equals_library_sdpa():
    H, D, n = 8, 64, 77
    q, K, V = f16((H, D)), f16((n, D)), f16((n, D))
    np.testing.assert_allclose(oracle.attend(q, K, V, 0.125), sdpa64(q, K, V, 0.125),
                               rtol=0, atol=1e-12)


def test_attend_identical_keys_give_mean_of_values():
    H, D, n = 4, 16, 9
    q, V = f16((H, D)), f16((n, D))
    K = np.repeat(f16((1, D)), n, axis=0)
    out = oracle.attend(q, K, V, 0.25)
    np.testing.assert_allclose(out, np.broadcast_to(V.astype(np.float64).mean(0), (H, D)),
                               rtol=0, atol=1e-14)


def test_attend_two_rows_closed_form():
    # logits (0, ln 3) -> weights (1/4, 3/4)
    q = np.array([[1.0, 0.0]])
    K = np.array([[0.0, 5.0], [math.log(3.0), -1.0]])
    V = np.array([[4.0, 8.0], [0.0, -4.0]])
    np.testing.assert_allclose(oracle.attend(q, K, V, 1.0), [[1.0, -1.0]], rtol=0, atol=1e-14)


def test_attend_union_order_and_split_merge():
    H, D, n = 8, 32, 50
    q, K, V = f16((H, D)), f16((n, D)), f16((n, D))
    scale = 1 / math.sqrt(D)
    full = oracle.attend(q, K, V, scale)
    perm = rng.permutation(n)
    np.testing.assert_allclose(oracle.attend(q, K[perm], V[perm], scale), full, rtol=0, atol=1e-13)
    # split into two parts and merge the parts by log-sum-exp weights
    from scipy.special import logsumexp
    a, b = perm[:17], perm[17:]
    z = scale * q.astype(np.float64) @ K.astype(np.float64).T           # [H, n]
    la, lb = logsumexp(z[:, a], axis=1), logsumexp(z[:, b], axis=1)
    oa, ob = oracle.attend(q, K[a], V[a], scale), oracle.attend(q, K[b], V[b], scale)
    wa = 1.0 / (1.0 + np.exp(lb - la))
    np.testing.assert_allclose(wa[:, None] * oa + (1 - wa)[:, None] * ob, full, rtol=0, atol=1e-13)


def _union_rows(raw_k, raw_v, raw_pos0, p, W, comp_k, comp_v, sel):
    lo = max(0, p - W + 1)
    K = [raw_k[lo - raw_pos0: p - raw_pos0 + 1]]
    V = [raw_v[lo - raw_pos0: p - raw_pos0 + 1]]
    if sel is not None:
        sel = [j for j in sel if j >= 0]
        K.append(comp_k[sel])
        V.append(comp_v[sel])
    return np.concatenate(K), np.concatenate(V)


@pytest.mark.parametrize("p", [0, 5, 31, 32, 200])
def test_decode_attend_equals_sdpa_over_window_and_selected_rows(p):
    H, D, W = 8, 64, 32
    raw_pos0 = max(0, p - 40)
    raw_k, raw_v = f16((p - raw_pos0 + 1, D)), f16((p - raw_pos0 + 1, D))
    comp_k, comp_v = f16((60, D)), f16((60, D))
    q = f16((H, D))
    sel = np.array([3, 7, -1, 12, 59, -1], dtype=np.int32)
    out = oracle.decode_attend(q, p, W, raw_k, raw_v, raw_pos0, comp_k, comp_v, sel, len(sel), 0.125)
    K, V = _union_rows(raw_k, raw_v, raw_pos0, p, W, comp_k, comp_v, sel)
    assert K.shape[0] == min(W, p + 1) + 4
    np.testing.assert_allclose(out, sdpa64(q, K, V, 0.125), rtol=0, atol=1e-12)
    # no selection list: rows 0..n_sel-1
    out_all = oracle.decode_attend(q, p, W, raw_k, raw_v, raw_pos0, comp_k, comp_v, None, 60, 0.125)
    K, V = _union_rows(raw_k, raw_v, raw_pos0, p, W, comp_k, comp_v, np.arange(60))
    np.testing.assert_allclose(out_all, sdpa64(q, K, V, 0.125), rtol=0, atol=1e-12)
    # window only
    out_w = oracle.decode_attend(q, p, W, raw_k, raw_v, raw_pos0, None, None, None, 0, 0.125)
    K, V = _union_rows(raw_k, raw_v, raw_pos0, p, W, None, None, None)
    np.testing.assert_allclose(out_w, sdpa64(q, K, V, 0.125), rtol=0, atol=1e-12)


def test_decode_attend_rejects_missing_window_rows():
    D = 8
    with pytest.raises(ValueError):
        oracle.decode_attend(f16((2, D)), 50, 32, f16((10, D)), f16((10, D)), 41, None, None, None, 0, 1.0)


def test_prefill_equals_masked_sdpa_all_rows():
    # ratio-128-like layer without indexer, at small sizes: every visible row attended
    H, D, W, r, T, P = 4, 32, 8, 4, 24, 20
    n_prior = min(W - 1, P)
    raw_k, raw_v = f16((n_prior + T, D)), f16((n_prior + T, D))
    n_comp = (P + T) // r
    comp_k, comp_v = f16((n_comp, D)), f16((n_comp, D))
    q = f16((T, H, D))
    out = oracle.prefill_attend(q, raw_k, raw_v, n_prior, W, comp_k, comp_v, None, P, r, 0.2)
    Kall = torch.tensor(np.concatenate([raw_k, comp_k]).astype(np.float64))
    Vall = torch.tensor(np.concatenate([raw_v, comp_v]).astype(np.float64))
    mask = torch.zeros(T, n_prior + T + n_comp, dtype=torch.bool)
    for i in range(T):
        p = P + i
        for t in range(max(0, p - W + 1), p + 1):
            mask[i, t - (P - n_prior)] = True
        for j in range(n_comp):
            mask[i, n_prior + T + j] = (j + 1) * r <= p + 1
    qt = torch.tensor(q.astype(np.float64)).permute(1, 0, 2)[None]          # [1, H, T, D]
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, Kall[None, None].expand(1, H, -1, -1), Vall[None, None].expand(1, H, -1, -1),
        attn_mask=mask[None, None], scale=0.2)
    np.testing.assert_allclose(out, o[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_prefill_one_token_equals_decode_and_is_causal():
    H, D, W, r, T, P, k = 4, 32, 16, 4, 12, 33, 5
    inst = synth.prefill_instance(seed=7, layer=2, H=H, D=D, window=W, ratio=r, d_idx=16, topk=k,
                                  P=P, T=T)
    res = oracle.prefill_chunk(inst)
    comp_k = np.concatenate([inst.comp_k.astype(np.float64), res["new_k"]])
    comp_v = np.concatenate([inst.comp_v.astype(np.float64), res["new_v"]])
    for i in [0, 5, T - 1]:
        p = P + i
        one = oracle.decode_attend(inst.q[i], p, W, inst.raw_k, inst.raw_v, P - inst.n_prior,
                                   comp_k, comp_v, res["sel"][i], k, inst.scale)
        np.testing.assert_allclose(res["out"][i], one, rtol=0, atol=1e-13)
    # perturbing the last token's q, k and v changes no earlier query's output
    inst.q = inst.q.copy()
    inst.raw_k = inst.raw_k.copy()
    inst.raw_v = inst.raw_v.copy()
    inst.q[-1] += np.float16(1.0)
    inst.raw_k[-1] += np.float16(1.0)
    inst.raw_v[-1] += np.float16(1.0)
    res2 = oracle.prefill_chunk(inst)
    np.testing.assert_array_equal(res2["out"][:-1], res["out"][:-1])
    assert not np.array_equal(res2["out"][-1], res["out"][-1])


def test_decode_step_pooled_history_matches_given_rows():
    # pooling the history inside the step equals giving the pooled rows as data
    inst = synth.decode_instance(seed=3, layer=2, H=8, D=32, window=16, ratio=4, d_idx=8, topk=6,
                                 p=71, pooled_history=True)
    a = oracle.decode_step(inst)
    assert a["n_vis"] == 18 and a["comp_k"].shape == (18, 32)
    ck, cv = oracle.compress_range(inst.raw_k, inst.raw_v, 0, inst.w, 4, 0, 18)
    np.testing.assert_array_equal(a["comp_k"], ck)
    np.testing.assert_array_equal(a["comp_v"], cv)
    K, V = _union_rows(inst.raw_k, inst.raw_v, 0, 71, 16, ck, cv, a["sel"])
    np.testing.assert_allclose(a["out"], sdpa64(inst.q, K, V, inst.scale), rtol=0, atol=1e-12)


# ---- generator ---------------------------------------------------------------------

def test_splitmix64_first_output():
    # published first output of SplitMix64 seeded with 0
    assert int(synth.raw_u64(0, 1)[0]) == 0xE220A8397B1DCDAF


def test_normals_moments_and_fp16_rounding():
    x = synth.normals(synth.stream_seed(0, 0, 1), 200000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    h = synth.normal_f16(0, 0, 1, (1000,))
    # RNE: every fp16 value is the nearest half to its double
    d = x[:1000]
    err = np.abs(h.astype(np.float64) - d)
    up = np.abs(np.nextafter(h, np.float16(np.inf)).astype(np.float64) - d)
    dn = np.abs(np.nextafter(h, np.float16(-np.inf)).astype(np.float64) - d)
    assert (err <= up).all() and (err <= dn).all()
