"""Per-layer device state and the decode / prefill steps, driven through the C ABI.

Layer schedule ("DS4 (DwarfStar 4)", Key Techniques, "KV attention
compression"): layers 0-1 attend the raw window only; even layers from 2
compress at ratio 4 and keep the indexer's top 512 rows; odd layers compress at
ratio 128 and attend every compressed row.

The KV state of one layer lives on the device, owned here (allocated through
torch): the raw window ring [W, D] (token p sits in slot p % W), the compressed
rows [cap, D], one indexer key per compressed row, and the compressor's running
state.  A decode step is, on the current stream: indexer_topk (ratio-4 layers),
compress_append of the new token (read from its ring slot) and attn_decode over
the ring and the kept rows.  Ratio-4 layers run the first two in one launch
(ds4a_indexer_topk_compress), ratio-128 layers the last two
(ds4a_compress_attn_decode), so every step is at most two dependent kernels.
"""
from __future__ import annotations

import copy
import math

import numpy as np
import torch

from . import ds4a

N_LAYERS = 43
N_HEADS = 64
HEAD_DIM = 128
WINDOW = 128
INDEX_DIM = 128
TOPK = 512


def layer_schedule(layer: int) -> tuple[int, int]:
    """(ratio, top_k) of a layer: ratio 0 = raw window only; top_k 0 = no indexer."""
    if layer < 2:
        return 0, 0
    if layer % 2 == 0:
        return 4, TOPK
    return 128, 0


def _dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DecodeLayer:
    """Device state of one layer for batch-1 decode, loaded from a DecodeInstance."""

    def __init__(self, inst, device="cuda", cap_extra: int = 0):
        self.inst = inst
        self.H, self.D, self.W = inst.H, inst.D, inst.window
        self.ratio, self.topk, self.p = inst.ratio, inst.topk, inst.p
        self.scale = 1.0 / math.sqrt(self.D)
        dev = torch.device(device)
        D, W = self.D, self.W
        p = self.p
        # raw window ring: token t in slot t % W
        self.ring_k = torch.zeros(W, D, dtype=torch.float16, device=dev)
        self.ring_v = torch.zeros(W, D, dtype=torch.float16, device=dev)
        lo = max(0, p - W + 1)
        pos = np.arange(lo, p + 1)
        rk, rv = inst.raw_k[pos - inst.raw_pos0], inst.raw_v[pos - inst.raw_pos0]
        slots = torch.from_numpy(pos % W).to(dev)
        self.ring_k[slots] = _dev(rk, dev)
        self.ring_v[slots] = _dev(rv, dev)
        self.n_win = len(pos)
        self.q = _dev(inst.q, dev)
        self.w = _dev(inst.w, dev)
        # pooled keys: the compressor also pools per-token indexer keys into the rows' keys
        self.pooled_keys = getattr(inst, "kidx_tok", None) is not None and inst.topk > 0
        d_state = 2 + 2 * D + (inst.d_idx if self.pooled_keys else 0)
        self.state = torch.zeros(d_state, dtype=torch.float32, device=dev)
        self.out = torch.empty(self.H, D, dtype=torch.float16, device=dev)
        self.n_vis = (p + 1) // self.ratio if self.ratio else 0
        if self.ratio:
            cap = max(1, self.n_vis + cap_extra)
            self.comp_k = torch.zeros(cap, D, dtype=torch.float16, device=dev)
            self.comp_v = torch.zeros(cap, D, dtype=torch.float16, device=dev)
            n_given = inst.comp_k.shape[0]
            if n_given:
                self.comp_k[:n_given] = _dev(inst.comp_k, dev)
                self.comp_v[:n_given] = _dev(inst.comp_v, dev)
        else:
            self.comp_k = self.comp_v = None
        if self.topk:
            # one indexer key per compressed row; rows past the given ones are filled as
            # advance() completes their blocks
            self.kidx = torch.zeros(max(1, self.n_vis + cap_extra), inst.d_idx, dtype=torch.float16, device=dev)
            if inst.kidx.shape[0]:
                self.kidx[: inst.kidx.shape[0]] = _dev(inst.kidx, dev)
            self.q_idx = _dev(inst.q_idx, dev)
            self.sel = torch.full((self.topk,), -1, dtype=torch.int32, device=dev)
            self.sel_n = torch.zeros(1, dtype=torch.int32, device=dev)
            nb = ds4a.ds4a_indexer_workspace_bytes(1, self.kidx.shape[0], self.topk)
            self.ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        else:
            self.kidx = self.q_idx = self.sel = self.sel_n = self.ws = None
        self.ki_tok = None
        if self.pooled_keys:
            self.ki_tok = _dev(inst.kidx_tok[p - inst.raw_pos0: p - inst.raw_pos0 + 1], dev)   # token p's key
        if self.ratio:
            # feed the compressor every raw token before p that it has not seen
            first = 0 if inst.pooled_history else (p // self.ratio) * self.ratio
            if p > first:
                a, b = first - inst.raw_pos0, p - inst.raw_pos0
                hk, hv = _dev(inst.raw_k[a:b], dev), _dev(inst.raw_v[a:b], dev)
                if self.pooled_keys:
                    ds4a.ds4a_compress_append_keys(hk, hv, _dev(inst.kidx_tok[a:b], dev), self.w, self.ratio, first,
                                                   self.state, self.comp_k, self.comp_v, self.kidx)
                else:
                    ds4a.ds4a_compress_append(hk, hv, self.w, self.ratio, first, self.state, self.comp_k,
                                              self.comp_v)
        self.slot = p % W

    def clone(self) -> "DecodeLayer":
        """An independent copy of the device state (same values, new buffers)."""
        c = copy.copy(self)
        for name, val in vars(self).items():
            if isinstance(val, torch.Tensor):
                setattr(c, name, val.clone())
        if c.ws is not None:
            c.ws.zero_()
        return c

    def bytes_touched(self) -> int:
        """Device bytes one decode step reads or writes (the algorithmic traffic)."""
        D = self.D
        b = 2 * self.H * D * 2                                  # q in, out
        b += 2 * self.n_win * D * 2                             # window K, V
        if self.ratio:
            b += 2 * D * 2 + D * 4 + (2 + 2 * D) * 4            # new token K, V; w; state
            n_rows = self.topk if self.topk else self.n_vis
            b += 2 * min(n_rows, self.n_vis) * D * 2            # kept compressed rows K, V
        if self.topk:
            b += self.n_vis * self.kidx.shape[1] * 2 + self.kidx.shape[1] * 2  # indexer keys, query
            b += self.topk * 4 * 2 + 4                          # kept indices written, read back
        if self.pooled_keys:
            b += self.kidx.shape[1] * (2 + 4)                   # the token's indexer key; its state
        return b

    def step(self, stream=None):
        """One decode step at position p (all inputs already resident).

        The indexer reads only the indexer keys (caller-supplied for every visible
        row), not the compressor's output, and the compressor reads only the new
        token: on ratio-4 layers one launch runs both.  A ratio-128 layer attends
        every row, and the compressor's update runs inside the attention launch.
        Under programmatic dependent launch the first kernel's input-only loads
        overlap the previous layer's attention.
        """
        for name, args in self._step_calls():
            getattr(ds4a, name)(*args, stream=stream)
        return self.out

    def advance(self, k, v, q, q_idx=None, kidx_row=None, stream=None, ki_tok=None):
        """Decode the next token: position p + 1.

        Appends the token's K and V (device [D] or [1, D] fp16) to the raw window
        ring, in slot (p + 1) % W, overwriting the token that leaves the window;
        takes the step's query q [H, D] and, on an indexer layer, its indexer query
        q_idx [d_idx]; then runs step() at the new position.  On an indexer layer a
        step that completes a block (p + 2 a multiple of the ratio) makes a new
        compressed row visible to its own query, so the row's indexer key kidx_row
        [d_idx] is required then.  The copies are stream-ordered device copies on
        `stream`, issued before the step's kernels.  Calls marshalled by bind()
        keep the position they were bound at: bind again after advancing.
        """
        p = self.p + 1
        n_vis, completes = self._check_next(p, q_idx, kidx_row, ki_tok)
        cur = torch.cuda.current_stream(self.q.device) if stream is None else stream
        slot = p % self.W
        with torch.cuda.stream(cur):
            self.ring_k[slot].copy_(k.reshape(-1), non_blocking=True)
            self.ring_v[slot].copy_(v.reshape(-1), non_blocking=True)
            self.q.copy_(q.reshape(self.q.shape), non_blocking=True)
            if self.topk:
                self.q_idx.copy_(q_idx.reshape(-1), non_blocking=True)
                if self.pooled_keys:
                    self.ki_tok.copy_(ki_tok.reshape(self.ki_tok.shape), non_blocking=True)
                elif completes:
                    self.kidx[n_vis - 1].copy_(kidx_row.reshape(-1), non_blocking=True)
        self._moved_to(p, n_vis)
        return self.step(stream=stream)

    def desc(self) -> "ds4a.DecodeLayerDesc":
        """The layer's ds4a_decode_layer_t (its persistent device arrays)."""
        return ds4a.decode_layer_desc(self.ring_k, self.ring_v, self.q, self.out, self.scale, self.ratio, self.w,
                                      self.state, self.comp_k, self.comp_v, self.topk, self.kidx, self.q_idx,
                                      self.sel, self.sel_n, self.ws, self.ki_tok)

    def _check_next(self, p, q_idx, kidx_row, ki_tok):
        n_vis = (p + 1) // self.ratio if self.ratio else 0
        if self.ratio and n_vis > self.comp_k.shape[0]:
            raise ValueError(f"advance: row {n_vis - 1} is past the compressed-row capacity {self.comp_k.shape[0]}")
        completes = bool(self.ratio) and (p + 1) % self.ratio == 0
        if self.topk:
            if q_idx is None:
                raise ValueError("advance: an indexer layer needs the step's indexer query")
            if self.pooled_keys and ki_tok is None:
                raise ValueError("advance: a layer that pools its indexer keys needs the token's key")
            if completes and kidx_row is None and not self.pooled_keys:
                raise ValueError(f"advance: position {p} completes row {n_vis - 1}, whose indexer key is required")
            if n_vis > self.kidx.shape[0]:
                raise ValueError("advance: past the indexer-key capacity")
        return n_vis, completes

    def _moved_to(self, p, n_vis):
        self.p, self.slot, self.n_vis = p, p % self.W, n_vis
        self.n_win = min(self.W, p + 1)

    def advance_host(self, k, v, q, q_idx=None, kidx_row=None, ki_tok=None, out=None, stream=None):
        """advance() from host memory through one C call (ds4a_decode_layer_step):
        k, v [D], q [H, D], q_idx, kidx_row and ki_tok [d_idx] are contiguous fp16 CPU
        tensors (page-locked for asynchronous copies).  The output is copied into `out`
        (an [H, D] fp16 CPU tensor, allocated when None) and returned once it is there."""
        p = self.p + 1
        n_vis, completes = self._check_next(p, q_idx, kidx_row, ki_tok)
        if out is None:
            out = torch.empty(self.H, self.D, dtype=torch.float16)
        ds4a.ds4a_decode_layer_step(self.desc(), p, k.reshape(-1), v.reshape(-1), q.reshape(-1),
                                    None if q_idx is None else q_idx.reshape(-1),
                                    kidx_row.reshape(-1) if (completes and self.topk and not self.pooled_keys) else None,
                                    None if ki_tok is None else ki_tok.reshape(-1), out, stream=stream)
        self._moved_to(p, n_vis)
        return out

    def bind_host(self, k, v, q, q_idx=None, out=None, ki_tok=None, stream=None):
        """The host-memory step at the current position marshalled once: a zero-argument
        callable that copies the host tensors in, runs the step, copies the output into
        `out` and waits (one C call).  For repeating one step, as bind()."""
        desc = self.desc()
        call = ds4a.bind("ds4a_decode_layer_step", desc, self.p, k.reshape(-1), v.reshape(-1), q.reshape(-1),
                         None if q_idx is None else q_idx.reshape(-1), None,
                         None if ki_tok is None else ki_tok.reshape(-1), out, stream=stream)

        def run():
            call()
            return out
        run.desc = desc          # keeps the descriptor alive with the call
        return run

    def bind(self, stream=None):
        """The decode step marshalled once (the layer's tensors are persistent): a
        zero-argument callable that issues the same launches as step(stream), without
        the binding's per-call Python argument checks."""
        calls = [ds4a.bind(name, *args, stream=stream) for name, args in self._step_calls()]

        def run():
            for c in calls:
                c()
            return self.out
        return run

    def _step_calls(self):
        """(binding function, arguments) of each launch of the step, in order."""
        new_k = self.ring_k[self.slot: self.slot + 1]
        new_v = self.ring_v[self.slot: self.slot + 1]
        win_k, win_v = self.ring_k[: self.n_win], self.ring_v[: self.n_win]
        if self.pooled_keys:
            # the compressor writes the key of a row this token completes and the indexer
            # ranks it in the same launch (its compressor CTA scores that row)
            return [("ds4a_indexer_topk_compress_keys", (self.q_idx, self.kidx, self.p, self.ratio, self.topk,
                                                         self.sel, self.sel_n, self.ws, new_k, new_v, self.ki_tok,
                                                         self.w, self.state, self.comp_k, self.comp_v)),
                    ("ds4a_attn_decode", (self.q, win_k, win_v, self.comp_k, self.comp_v, self.sel, self.topk,
                                          self.scale, self.out))]
        if self.topk:
            return [("ds4a_indexer_topk_compress", (self.q_idx, self.kidx, self.p, self.ratio, self.topk, self.sel,
                                                    self.sel_n, self.ws, new_k, new_v, self.w, self.state, self.comp_k,
                                                    self.comp_v)),
                    ("ds4a_attn_decode", (self.q, win_k, win_v, self.comp_k, self.comp_v, self.sel, self.topk,
                                          self.scale, self.out))]
        if self.ratio:
            return [("ds4a_compress_attn_decode", (new_k, new_v, self.w, self.ratio, self.p, self.state, self.comp_k,
                                                   self.comp_v, self.q, win_k, win_v, self.scale, self.out))]
        return [("ds4a_attn_decode", (self.q, win_k, win_v, self.comp_k, self.comp_v, None, self.n_vis, self.scale,
                                      self.out))]


class PrefillLayer:
    """Device state of one layer for one prefill chunk, loaded from a PrefillInstance."""

    def __init__(self, inst, device="cuda"):
        self.inst = inst
        dev = torch.device(device)
        self.T, self.H, self.D = inst.T, inst.H, inst.D
        self.P, self.ratio, self.topk, self.W = inst.P, inst.ratio, inst.topk, inst.window
        self.n_prior = inst.n_prior
        self.scale = 1.0 / math.sqrt(self.D)
        self.raw_k = _dev(inst.raw_k, dev)
        self.raw_v = _dev(inst.raw_v, dev)
        self.q = _dev(inst.q, dev)
        self.w = _dev(inst.w, dev)
        self.out = torch.empty(self.T, self.H, self.D, dtype=torch.float16, device=dev)
        self.state = torch.zeros(2 + 2 * self.D, dtype=torch.float32, device=dev)
        if self.ratio:
            n_end = (self.P + self.T) // self.ratio
            self.comp_k = torch.zeros(n_end, self.D, dtype=torch.float16, device=dev)
            self.comp_v = torch.zeros(n_end, self.D, dtype=torch.float16, device=dev)
            n_given = inst.comp_k.shape[0]
            if n_given:
                self.comp_k[:n_given] = _dev(inst.comp_k, dev)
                self.comp_v[:n_given] = _dev(inst.comp_v, dev)
            # the prefix's open block (if any) is fed before the chunk
            first = (self.P // self.ratio) * self.ratio
            if self.P > first:
                a, b = first - (self.P - self.n_prior), self.n_prior
                ds4a.ds4a_compress_append(self.raw_k[a:b], self.raw_v[a:b], self.w, self.ratio, first,
                                          self.state, self.comp_k, self.comp_v)
        else:
            self.comp_k = self.comp_v = None
        if self.topk:
            self.kidx = _dev(inst.kidx, dev)
            self.q_idx = _dev(inst.q_idx, dev)
            self.sel = torch.full((self.T, self.topk), -1, dtype=torch.int32, device=dev)
            self.sel_n = torch.zeros(self.T, dtype=torch.int32, device=dev)
            nb = ds4a.ds4a_indexer_workspace_bytes(self.T, self.kidx.shape[0], self.topk)
            self.ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        else:
            self.kidx = self.q_idx = self.sel = self.sel_n = self.ws = None

    def step(self, stream=None):
        """compress_append(chunk) -> indexer_topk(all queries) -> attn_prefill."""
        if self.ratio:
            ds4a.ds4a_compress_append(self.raw_k[self.n_prior:], self.raw_v[self.n_prior:], self.w, self.ratio,
                                      self.P, self.state, self.comp_k, self.comp_v, stream=stream)
        if self.topk:
            ds4a.ds4a_indexer_topk(self.q_idx, self.kidx, self.P, self.ratio, self.topk, self.sel, self.sel_n,
                                   self.ws, stream=stream)
        ds4a.ds4a_attn_prefill(self.q, self.raw_k, self.raw_v, self.n_prior, self.W, self.comp_k, self.comp_v,
                               self.sel, self.P, self.ratio, self.scale, self.out, stream=stream)
        return self.out


class PrefillStack:
    """One prefill chunk through a stack of layers, each with its own schedule
    (layer_schedule: window only, ratio 4 + indexer top-512, ratio 128) and its own
    device state.  "DS4 (DwarfStar 4)", Architecture, "Whole-model graph execution":
    prefill runs the model's layers over chunks of tokens (2048 by default)."""

    def __init__(self, instances, device="cuda"):
        self.layers = [PrefillLayer(inst, device) for inst in instances]

    def step(self, stream=None):
        """Every layer's compress_append -> indexer_topk -> attn_prefill, layer after layer."""
        for L in self.layers:
            L.step(stream=stream)
        return [L.out for L in self.layers]


class BatchedDecodeLayer:
    """B independent decode sessions of one layer, stepped together: one launch of
    each batched kernel serves every session ("DwarfStar (ds4) Deep Dive",
    Step-by-Step Tutorial, "Start the Server": --batched-session 16).

    Built from one DecodeInstance per session (the same layer shape and schedule,
    any positions).  Device state is batched along a leading session axis: rings
    [B, W, D], compressed rows [B, cap, D], indexer keys [B, cap, d_idx], compressor
    states [B, 2 + 2D], positions pos [B] (int64, device memory).
    """

    def __init__(self, instances, device="cuda", cap_extra: int = 0):
        for inst in instances[1:]:
            if not np.array_equal(inst.w, instances[0].w):
                raise ValueError("BatchedDecodeLayer: the sessions of one layer share its compressor score weights")
        singles = [DecodeLayer(inst, device=device, cap_extra=0) for inst in instances]
        L0 = singles[0]
        for L in singles:
            if (L.H, L.D, L.W, L.ratio, L.topk) != (L0.H, L0.D, L0.W, L0.ratio, L0.topk) or L.pooled_keys:
                raise ValueError("BatchedDecodeLayer: sessions must share the layer's shape and schedule")
        self.B = len(singles)
        self.H, self.D, self.W, self.ratio, self.topk = L0.H, L0.D, L0.W, L0.ratio, L0.topk
        self.scale = L0.scale
        dev = torch.device(device)
        self.p_host = [L.p for L in singles]
        self.pos = torch.tensor(self.p_host, dtype=torch.int64, device=dev)
        self.ring_k = torch.stack([L.ring_k for L in singles])
        self.ring_v = torch.stack([L.ring_v for L in singles])
        self.q = torch.stack([L.q for L in singles])
        self.w = L0.w
        self.state = torch.stack([L.state for L in singles])
        self.out = torch.empty_like(self.q)
        self.cap = 0
        self.comp_k = self.comp_v = self.kidx = self.q_idx = self.sel = self.sel_n = self.ws = None
        if self.ratio:
            self.cap = max(1, max(L.n_vis for L in singles) + cap_extra)
            self.comp_k = torch.zeros(self.B, self.cap, self.D, dtype=torch.float16, device=dev)
            self.comp_v = torch.zeros_like(self.comp_k)
            for s, L in enumerate(singles):
                n = min(L.comp_k.shape[0], self.cap)
                self.comp_k[s, :n] = L.comp_k[:n]
                self.comp_v[s, :n] = L.comp_v[:n]
        if self.topk:
            d_idx = L0.kidx.shape[1]
            self.kidx = torch.zeros(self.B, self.cap, d_idx, dtype=torch.float16, device=dev)
            for s, L in enumerate(singles):
                n = min(L.kidx.shape[0], self.cap)
                self.kidx[s, :n] = L.kidx[:n]
            self.q_idx = torch.stack([L.q_idx for L in singles])
            self.sel = torch.full((self.B, self.topk), -1, dtype=torch.int32, device=dev)
            self.sel_n = torch.zeros(self.B, dtype=torch.int32, device=dev)
            self.ws = torch.zeros(ds4a.ds4a_decode_batched_workspace_bytes(self.B, self.cap), dtype=torch.uint8,
                                  device=dev)

    def clone(self) -> "BatchedDecodeLayer":
        c = copy.copy(self)
        for name, val in vars(self).items():
            if isinstance(val, torch.Tensor):
                setattr(c, name, val.clone())
        c.p_host = list(self.p_host)
        if c.ws is not None:
            c.ws.zero_()
        return c

    def bytes_touched(self) -> int:
        """Device bytes one batched step reads or writes (the sum over the sessions)."""
        D, b = self.D, 0
        for p in self.p_host:
            n_win = min(self.W, p + 1)
            n_vis = min((p + 1) // self.ratio, self.cap) if self.ratio else 0
            b += 2 * self.H * D * 2 + 2 * n_win * D * 2 + 8
            if self.ratio:
                b += 2 * D * 2 + D * 4 + (2 + 2 * D) * 4
                b += 2 * (min(self.topk, n_vis) if self.topk else n_vis) * D * 2
            if self.topk:
                b += n_vis * self.kidx.shape[2] * 2 + self.kidx.shape[2] * 2 + self.topk * 4 * 2 + 4
        return b

    def _step_calls(self):
        if self.topk:
            return [("ds4a_indexer_topk_compress_batched", (self.q_idx, self.kidx, self.pos, self.ratio, self.topk,
                                                            self.sel, self.sel_n, self.ws, self.ring_k, self.ring_v,
                                                            self.w, self.state, self.comp_k, self.comp_v)),
                    ("ds4a_attn_decode_batched", (self.q, self.ring_k, self.ring_v, self.pos, self.comp_k,
                                                  self.comp_v, self.sel, self.ratio, self.scale, self.out))]
        if self.ratio:
            return [("ds4a_compress_attn_decode_batched", (self.w, self.ratio, self.state, self.comp_k, self.comp_v,
                                                           self.q, self.ring_k, self.ring_v, self.pos, self.scale,
                                                           self.out))]
        return [("ds4a_attn_decode_batched", (self.q, self.ring_k, self.ring_v, self.pos, None, None, None, 0,
                                              self.scale, self.out))]

    def step(self, stream=None):
        """One decode step of every session at its position pos[s] (inputs resident)."""
        for name, args in self._step_calls():
            getattr(ds4a, name)(*args, stream=stream)
        return self.out

    def bind(self, stream=None):
        """The step marshalled once (see DecodeLayer.bind)."""
        calls = [ds4a.bind(name, *args, stream=stream) for name, args in self._step_calls()]

        def run():
            for c in calls:
                c()
            return self.out
        return run

    def advance(self, k, v, q, q_idx=None, kidx_rows=None, stream=None):
        """Every session decodes its next token: k, v [B, D] go to ring slot
        (pos + 1) % W of each session, q [B, H, D] and q_idx [B, d_idx] are the steps'
        queries; kidx_rows [B, d_idx] holds the indexer key of the row each session's
        token completes (rows of sessions that complete none are ignored).  The
        positions advance on the host and on the device."""
        p_new = [p + 1 for p in self.p_host]
        if self.ratio and max((p + 1) // self.ratio for p in p_new) > self.cap:
            raise ValueError("advance: a session's rows would pass the capacity")
        cur = torch.cuda.current_stream(self.q.device) if stream is None else stream
        dev = self.q.device
        sess = torch.arange(self.B, device=dev)
        slots = torch.tensor([p % self.W for p in p_new], dtype=torch.int64, device=dev)
        with torch.cuda.stream(cur):
            self.ring_k[sess, slots] = k
            self.ring_v[sess, slots] = v
            self.q.copy_(q, non_blocking=True)
            if self.topk:
                self.q_idx.copy_(q_idx, non_blocking=True)
                done = [s for s, p in enumerate(p_new) if (p + 1) % self.ratio == 0]
                if done:
                    if kidx_rows is None:
                        raise ValueError("advance: sessions completing a row need its indexer key")
                    rows = torch.tensor([(p_new[s] + 1) // self.ratio - 1 for s in done], dtype=torch.int64, device=dev)
                    idx = torch.tensor(done, dtype=torch.int64, device=dev)
                    self.kidx[idx, rows] = kidx_rows[idx]
            self.pos.add_(1)
        self.p_host = p_new
        return self.step(stream=stream)
