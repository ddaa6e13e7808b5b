"""Parity criteria between the CUDA path and the oracle.

Outputs (fp16 result vs fp64 oracle): max |g - r| <= 2e-3 over every element AND
max |g - r| / max |r| <= 1e-2 (normwise relative error of the call).
Indices: bit-exact; the only tolerated difference is a swap among rows whose
oracle score (rounded to binary32, the precision both sides rank in) lies within
1e-6 relative of the k-th kept score.
"""
import numpy as np

ATOL = 2e-3
RTOL_NORM = 1e-2
TIE_REL = 1e-6


def check_out(gpu, ref, what="out"):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - r).max() if g.size else 0.0
    scale = np.abs(r).max() if r.size else 1.0
    assert err <= ATOL, f"{what}: max abs err {err:.3e} > {ATOL}"
    assert err <= RTOL_NORM * scale, f"{what}: normwise rel err {err / scale:.3e} > {RTOL_NORM}"
    return err


def check_sel(gpu_idx, ref_idx, scores, k, what="sel"):
    """gpu_idx / ref_idx: kept rows (ascending, padding dropped); scores: oracle scores (fp64)."""
    g = np.asarray([x for x in gpu_idx if x >= 0], dtype=np.int64)
    r = np.asarray([x for x in ref_idx if x >= 0], dtype=np.int64)
    assert len(g) == len(r), (what, len(g), len(r))
    assert (np.diff(g) > 0).all(), f"{what}: not strictly ascending"
    if np.array_equal(g, r):
        return 0
    s32 = np.asarray(scores, dtype=np.float32).astype(np.float64)
    kth = np.sort(s32[r])[0]
    band = TIE_REL * abs(kth)
    diff = np.setxor1d(g, r)
    bad = [j for j in diff if abs(s32[j] - kth) > band]
    assert not bad, f"{what}: {len(diff)} differing rows, {len(bad)} outside the tie band"
    return len(diff)


def check_sel_rounded_keys(gpu_idx, ref_idx, q, keys, what="sel"):
    """Kept rows ranked by keys that the GPU rounds to fp16 (pooled indexer keys) and the
    oracle keeps in fp64.  Rounding a key component to fp16 moves it by at most half an
    ulp, 2^-11 of its magnitude, so row j's score may move by up to
    b_j = 2^-11 * sum_c |q_c keys_jc| (with 5% slack, plus the binary32 ranking
    precision).  The kept lists must have the same length and be ascending; a row kept
    by one side only must have an oracle score within b_j + b_kth of the k-th kept
    score.  Returns the number of differing rows."""
    g = np.asarray([x for x in gpu_idx if x >= 0], dtype=np.int64)
    r = np.asarray([x for x in ref_idx if x >= 0], dtype=np.int64)
    assert len(g) == len(r), (what, len(g), len(r))
    assert (np.diff(g) > 0).all(), f"{what}: not strictly ascending"
    if np.array_equal(g, r):
        return 0
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    s = keys @ q
    b = 1.05 * 2.0 ** -11 * (np.abs(keys) @ np.abs(q))
    kth = int(r[np.argmin(s[r])])
    diff = np.setxor1d(g, r)
    bad = [j for j in diff if abs(s[j] - s[kth]) > b[j] + b[kth] + TIE_REL * abs(s[kth])]
    assert not bad, f"{what}: {len(diff)} differing rows, {len(bad)} outside the fp16 key-rounding band"
    return len(diff)
