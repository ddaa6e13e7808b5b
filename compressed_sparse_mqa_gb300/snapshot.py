"""Snapshot and restore of the decode state of a stack of layers, as one blob.

"DS4 (DwarfStar 4)", Key Techniques, "KV cache with disk as first-class
citizen": the KV cache has three tiers (the raw sliding window, the compressed
rows pooled at ratio boundaries, and serialized snapshots on disk), and a
snapshot carries the per-layer compressed row counts, the raw sliding-window
rows and the compressor/indexer frontiers.  Design Decisions, "Innovation: disk
KV as first-class citizen": a cold save trims 32 tail tokens and aligns to
2048-token chunk boundaries, continued saves write at alignment frontiers.

What one layer's record holds (everything a later decode step reads that an
earlier step wrote or the caller supplied as cache):
  * the position p of the last token fed, the layer's shape and schedule;
  * the raw window ring [W, D] K and V, token t in slot t % W;
  * the compressor frontier: its running state [2 + 2D] fp32 (the open block's
    running max, sum and weighted K/V sums) -- the open block's tokens need not
    be kept, the state stands for them;
  * the compressed rows 0 .. n_rows-1 (K and V) with n_rows = floor((p+1)/r);
  * the indexer frontier: the indexer keys of those rows.
The indexer workspace, the kept-row list and the queries are per-step scratch
and outputs, not state.

Blob layout (little-endian): a 16-byte header "DS4ASNAP", u32 version, u32
layer count; then per layer a 64-byte record header (seven i32: ratio, topk, H,
D, W, d_idx, pooled (1 when the layer's compressor pools indexer keys, whose
weighted sum then extends the state by d_idx floats); then i64 p, i64 n_rows;
zero padding) followed by the arrays, each padded to a 16-byte multiple: ring K,
ring V (fp16), state (fp32), compressed K, compressed V (fp16), indexer keys
(fp16, indexer layers only).
"""
from __future__ import annotations

import struct

import numpy as np
import torch

MAGIC = b"DS4ASNAP"
VERSION = 1
_HDR = struct.Struct("<8sII")                 # 16 bytes
_REC = struct.Struct("<7iqq")                 # 44 bytes, padded to 64
_REC_BYTES = 64

# "Innovation: disk KV as first-class citizen": saves land on 2048-token chunk
# boundaries, a cold save after trimming 32 tail tokens
CHUNK_ALIGN = 2048
COLD_TRIM = 32


def save_frontier(n_tokens: int, cold: bool = True, align: int = CHUNK_ALIGN, trim: int = COLD_TRIM) -> int:
    """The token count a save of an n_tokens-long session keeps: the largest multiple of
    `align` not above n_tokens - trim (cold save) or n_tokens (continued save)."""
    n = n_tokens - (trim if cold else 0)
    return max(0, n // align) * align


def _pad16(n: int) -> int:
    return (n + 15) // 16 * 16


def _arrays(L):
    """The record's arrays of one layer, as contiguous host numpy arrays."""
    n_rows = (L.p + 1) // L.ratio if L.ratio else 0
    arrs = [L.ring_k, L.ring_v, L.state]
    if L.ratio:
        arrs += [L.comp_k[:n_rows], L.comp_v[:n_rows]]
    if L.topk:
        arrs += [L.kidx[:n_rows]]
    return n_rows, [a.detach().contiguous().cpu().numpy() for a in arrs]


def _pooled(L) -> bool:
    return bool(getattr(L, "pooled_keys", False))


def snapshot(layers) -> bytes:
    """One blob holding the decode state of every layer (DecodeLayer objects, or any
    objects with the same fields).  Reads the device state after the current stream's
    work: call it between steps."""
    if torch.cuda.is_available():
        torch.cuda.current_stream().synchronize()
    parts = [_HDR.pack(MAGIC, VERSION, len(layers))]
    for L in layers:
        n_rows, arrs = _arrays(L)
        d_idx = L.kidx.shape[1] if L.topk else 0
        rec = _REC.pack(L.ratio, L.topk, L.H, L.D, L.W, d_idx, int(_pooled(L)), L.p, n_rows)
        parts.append(rec + b"\0" * (_REC_BYTES - len(rec)))
        for a in arrs:
            b = a.tobytes()
            parts.append(b + b"\0" * (_pad16(len(b)) - len(b)))
    return b"".join(parts)


class SnapshotError(ValueError):
    pass


def _take(blob: bytes, off: int, n: int) -> tuple[bytes, int]:
    if off + n > len(blob):
        raise SnapshotError("snapshot: blob is truncated")
    return blob[off:off + n], off + _pad16(n)


def restore(blob: bytes, layers) -> None:
    """Write the state in `blob` into `layers` (same count, shapes and schedule as the
    layers the blob was taken from; capacities at least the blob's row counts).  The
    copies are stream-ordered on the current stream; the layers' positions become the
    blob's.  Raises SnapshotError on a malformed or mismatching blob and leaves the
    layers unchanged in that case (every record is checked before any is written)."""
    if len(blob) < _HDR.size:
        raise SnapshotError("snapshot: blob is truncated")
    magic, version, n_layers = _HDR.unpack_from(blob, 0)
    if magic != MAGIC:
        raise SnapshotError("snapshot: not a ds4a snapshot")
    if version != VERSION:
        raise SnapshotError(f"snapshot: version {version}, expected {VERSION}")
    if n_layers != len(layers):
        raise SnapshotError(f"snapshot: {n_layers} layers in the blob, {len(layers)} given")
    off = _HDR.size
    plan = []
    for i, L in enumerate(layers):
        rec, off = _take(blob, off, _REC_BYTES)
        ratio, topk, H, D, W, d_idx, pooled, p, n_rows = _REC.unpack_from(rec, 0)
        mine = (L.ratio, L.topk, L.H, L.D, L.W, L.kidx.shape[1] if L.topk else 0, int(_pooled(L)))
        if (ratio, topk, H, D, W, d_idx, pooled) != mine:
            raise SnapshotError(f"snapshot: layer {i} is (ratio, topk, H, D, W, d_idx, pooled) = "
                                f"{(ratio, topk, H, D, W, d_idx, pooled)}, the target is {mine}")
        if p < 0 or n_rows != ((p + 1) // ratio if ratio else 0):
            raise SnapshotError(f"snapshot: layer {i} row count {n_rows} does not match position {p}")
        if ratio and (n_rows > L.comp_k.shape[0] or (topk and n_rows > L.kidx.shape[0])):
            raise SnapshotError(f"snapshot: layer {i} has {n_rows} rows, more than the target's capacity")
        specs = [(L.ring_k, (W, D), np.float16), (L.ring_v, (W, D), np.float16),
                 (L.state, (2 + 2 * D + (d_idx if pooled else 0),), np.float32)]
        if ratio:
            specs += [(L.comp_k, (n_rows, D), np.float16), (L.comp_v, (n_rows, D), np.float16)]
        if topk:
            specs += [(L.kidx, (n_rows, d_idx), np.float16)]
        arrays = []
        for dst, shape, dt in specs:
            nbytes = int(np.prod(shape)) * np.dtype(dt).itemsize
            raw, off = _take(blob, off, nbytes)
            arrays.append((dst, np.frombuffer(raw, dtype=dt).reshape(shape)))
        plan.append((L, p, n_rows, arrays))
    if off != _pad16(len(blob)) and off != len(blob):
        raise SnapshotError("snapshot: trailing bytes after the last layer")
    for L, p, n_rows, arrays in plan:
        for dst, a in arrays:
            src = torch.from_numpy(a.copy())
            dst[: a.shape[0]].copy_(src.view(dst.dtype) if src.dtype != dst.dtype else src, non_blocking=False)
        L.p = p
        L.n_vis = n_rows
        L.slot = p % L.W
        L.n_win = min(L.W, p + 1)
