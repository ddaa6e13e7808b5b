"""Host-side tests of the C ABI (no GPU needed).

The library must load, export every entry point include/*.h declares, and
reject bad arguments before any CUDA call is made (so these run on a CPU-only
machine: the calls below return an argument error before touching a device).
"""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT

HEADERS = glob.glob(os.path.join(ROOT, "include", "*.h"))


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(ds4a_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_four_path_calls():
    names = declared_functions()
    for n in ["ds4a_compress_append", "ds4a_indexer_topk", "ds4a_attn_decode", "ds4a_attn_prefill"]:
        assert n in names


def test_library_exports_every_declared_symbol(ds4a_lib):
    L = ctypes.CDLL(ds4a_lib.LIB_PATH)
    for n in declared_functions():
        assert hasattr(L, n), n
    assert set(declared_functions()) <= set(ds4a_lib.EXPORTED) | set(declared_functions())


def test_status_strings(ds4a_lib):
    L = ds4a_lib.lib()
    assert L.ds4a_status_str(0) == b"ok"
    assert L.ds4a_status_str(7).startswith(b"row index")
    assert L.ds4a_status_str(99) == b"unknown status"


FAKE = 0x10000          # never dereferenced: every call below fails validation first
ARG, UNSUP, WS, CAP = 1, 3, 6, 2


def test_compress_append_validation(ds4a_lib):
    L = ds4a_lib.lib()
    f = L.ds4a_compress_append
    # negative n_new, bad ratio, bad head_dim, null pointer, misaligned k, capacity
    assert f(FAKE, FAKE, -1, 128, FAKE, 4, 0, FAKE, FAKE, FAKE, 10, None) == ARG
    assert f(FAKE, FAKE, 1, 128, FAKE, 0, 0, FAKE, FAKE, FAKE, 10, None) == ARG
    assert f(FAKE, FAKE, 1, 100, FAKE, 4, 0, FAKE, FAKE, FAKE, 10, None) == UNSUP
    assert f(FAKE, FAKE, 1, 128, FAKE, 2048, 0, FAKE, FAKE, FAKE, 10, None) == UNSUP
    assert f(None, FAKE, 1, 128, FAKE, 4, 0, FAKE, FAKE, FAKE, 10, None) == ARG
    assert f(FAKE + 8, FAKE, 1, 128, FAKE, 4, 0, FAKE, FAKE, FAKE, 10, None) == ARG
    assert f(FAKE, FAKE, 8, 128, FAKE, 4, 36, FAKE, FAKE, FAKE, 10, None) == CAP   # rows up to 11 > 10
    assert f(None, None, 0, 128, None, 4, 0, None, None, None, 0, None) == 0       # n_new = 0: no-op


def test_indexer_validation(ds4a_lib):
    L = ds4a_lib.lib()
    f = L.ds4a_indexer_topk
    nb = L.ds4a_indexer_workspace_bytes(1, 8192, 512)
    assert nb >= 8192 * 4
    assert f(FAKE, 1, FAKE, 8192, 128, 32768, 4, 0, FAKE, FAKE, FAKE, nb, None) == ARG      # k = 0
    assert f(FAKE, 1, FAKE, 8192, 100, 32768, 4, 512, FAKE, FAKE, FAKE, nb, None) == UNSUP  # d_idx
    assert f(FAKE, 1, FAKE, 8192, 128, 32768, 4, 4096, FAKE, FAKE, FAKE, nb, None) == UNSUP  # k too big
    assert f(FAKE, 1, FAKE, 8192, 128, 32768, 0, 512, FAKE, FAKE, FAKE, nb, None) == ARG    # ratio
    assert f(FAKE, 1, FAKE, 8192, 128, 32768, 4, 512, FAKE, FAKE, None, nb, None) == WS     # no ws
    assert f(FAKE, 1, FAKE, 8192, 128, 32768, 4, 512, FAKE, FAKE, FAKE, nb - 1, None) == WS
    assert f(FAKE + 4, 1, FAKE, 8192, 128, 32768, 4, 512, FAKE, FAKE, FAKE, nb, None) == ARG
    assert f(None, 0, None, 0, 128, 0, 4, 512, None, None, None, 0, None) == 0            # n_q = 0


def test_indexer_topk_compress_validation(ds4a_lib):
    L = ds4a_lib.lib()
    f = L.ds4a_indexer_topk_compress
    nb = L.ds4a_indexer_workspace_bytes(1, 8192, 512)

    def call(**kw):
        a = dict(q=FAKE, kidx=FAKE, n_rows=8192, d_idx=128, q_pos=32768, ratio=4, k=512, out=FAKE, out_n=FAKE,
                 ws=FAKE, nb=nb, k_new=FAKE, v_new=FAKE, head_dim=128, w=FAKE, state=FAKE, ck=FAKE, cv=FAKE,
                 cap=9000)
        a.update(kw)
        return f(a["q"], a["kidx"], a["n_rows"], a["d_idx"], a["q_pos"], a["ratio"], a["k"], a["out"], a["out_n"],
                 a["ws"], a["nb"], a["k_new"], a["v_new"], a["head_dim"], a["w"], a["state"], a["ck"], a["cv"],
                 a["cap"], None)
    assert call(k=0) == ARG
    assert call(ratio=0) == ARG
    assert call(d_idx=100) == UNSUP
    assert call(head_dim=100) == UNSUP
    assert call(ratio=2048) == UNSUP
    assert call(k_new=None) == ARG
    assert call(state=None) == ARG
    assert call(k_new=FAKE + 8) == ARG          # the token rows must be 16-byte aligned
    assert call(q=FAKE + 4) == ARG
    assert call(ws=None) == WS
    assert call(nb=nb - 1) == WS
    assert call(q_pos=32771, cap=8192) == CAP   # position 32771 completes row 8192 (rows 0 .. 8191 fit)


def test_compress_attn_decode_validation(ds4a_lib):
    L = ds4a_lib.lib()
    f = L.ds4a_compress_attn_decode

    def call(**kw):
        a = dict(k_new=FAKE, v_new=FAKE, w=FAKE, ratio=128, pos=131071, state=FAKE, ck=FAKE, cv=FAKE, cap=1024,
                 q=FAKE, H=64, D=128, wk=FAKE, wv=FAKE, n_win=128, out=FAKE)
        a.update(kw)
        return f(a["k_new"], a["v_new"], a["w"], a["ratio"], a["pos"], a["state"], a["ck"], a["cv"], a["cap"],
                 a["q"], a["H"], a["D"], a["wk"], a["wv"], a["n_win"], ctypes.c_float(0.088), a["out"], None)
    assert call(ratio=0) == ARG
    assert call(pos=-1) == ARG
    assert call(H=12) == UNSUP
    assert call(D=96) == UNSUP
    assert call(ratio=2048) == UNSUP
    assert call(n_win=0) == ARG
    assert call(state=None) == ARG
    assert call(out=None) == ARG
    assert call(k_new=FAKE + 8) == ARG          # the token rows must be 16-byte aligned
    assert call(ck=FAKE + 8) == ARG
    assert call(cap=1023) == CAP                # position 131071 completes row 1023


def test_attn_decode_validation(ds4a_lib):
    L = ds4a_lib.lib()
    f = L.ds4a_attn_decode
    s = ctypes.c_float(0.088)
    assert f(FAKE, 64, 96, FAKE, FAKE, 128, FAKE, FAKE, 100, FAKE, 512, s, FAKE, None, 0, None) == UNSUP
    assert f(FAKE, 60, 128, FAKE, FAKE, 128, FAKE, FAKE, 100, FAKE, 512, s, FAKE, None, 0, None) == UNSUP
    assert f(FAKE, 128, 128, FAKE, FAKE, 128, FAKE, FAKE, 100, FAKE, 512, s, FAKE, None, 0, None) == UNSUP
    assert f(FAKE, 64, 128, FAKE, FAKE, 0, FAKE, FAKE, 100, FAKE, 512, s, FAKE, None, 0, None) == ARG
    assert f(FAKE, 64, 128, FAKE, FAKE, 128, None, FAKE, 100, FAKE, 512, s, FAKE, None, 0, None) == ARG
    # sel = NULL means rows 0..n_sel-1: n_sel may not exceed n_comp
    assert f(FAKE, 64, 128, FAKE, FAKE, 128, FAKE, FAKE, 100, None, 101, s, FAKE, None, 0, None) == ARG
    assert f(FAKE, 64, 128, FAKE + 8, FAKE, 128, FAKE, FAKE, 100, None, 10, s, FAKE, None, 0, None) == ARG
    # n_win + n_sel must fit in an int (the kernel's row count)
    assert f(FAKE, 64, 128, FAKE, FAKE, 128, FAKE, FAKE, 100, FAKE, 2**31 - 100, s, FAKE, None, 0,
             None) == UNSUP


def test_noalloc_indexer_validation(ds4a_lib):
    """The allocation-free indexer's limit counts the rows the query sees: more rows than
    its scratch holds are refused only when the position makes them visible."""
    L = ctypes.CDLL(ds4a_lib.LIB_PATH)
    f = L.ds4a_indexer_topk_noalloc
    P, I, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    f.argtypes = [P, P, LL, I, LL, I, I, P, P, P]
    f.restype = I
    assert f(FAKE, FAKE, 70000, 128, 4 * 70000, 4, 512, FAKE, FAKE, None) == WS     # 70000 visible
    assert f(FAKE, FAKE, 65537, 128, 4 * 65537, 4, 512, FAKE, FAKE, None) == WS
    assert f(FAKE, FAKE, 70000, 128, 4 * 60000, 4, 0, FAKE, FAKE, None) == ARG      # 60000 visible, bad k
    assert f(FAKE, FAKE, 70000, 100, 4 * 60000, 4, 512, FAKE, FAKE, None) == UNSUP  # d_idx
    assert f(FAKE + 4, FAKE, 70000, 128, 4 * 60000, 4, 512, FAKE, FAKE, None) == ARG  # misaligned query


def test_attn_prefill_validation(ds4a_lib):
    L = ds4a_lib.lib()
    f = L.ds4a_attn_prefill
    s = ctypes.c_float(0.088)
    # n_prior must cover the window: min(window-1, q_pos0) rows
    assert f(FAKE, 16, 64, 128, FAKE, FAKE, 100, 128, FAKE, FAKE, 10, None, 0, 1000, 4, s, FAKE, None, 0,
             None) == ARG
    assert f(FAKE, 16, 64, 128, FAKE, FAKE, 20, 128, FAKE, FAKE, 10, None, 0, 10, 4, s, FAKE, None, 0,
             None) == ARG   # n_prior > q_pos0
    assert f(FAKE, 16, 64, 128, FAKE, FAKE, 127, 128, FAKE, FAKE, 10, FAKE, 0, 1000, 4, s, FAKE, None, 0,
             None) == ARG   # sel with k_stride 0
    assert f(FAKE, 16, 64, 64 + 8, FAKE, FAKE, 127, 128, FAKE, FAKE, 10, None, 0, 1000, 4, s, FAKE, None, 0,
             None) == UNSUP
    assert f(None, 0, 64, 128, None, None, 0, 128, None, None, 0, None, 0, 0, 4, s, None, None, 0,
             None) == 0     # T = 0: no-op


def test_binding_refuses_host_tensors(ds4a_lib):
    """The product path has no CPU fallback: the binding refuses host tensors before any
    C call (plain and one-launch decode calls, and the marshalled-once form)."""
    import torch
    H, D, W = 8, 64, 32
    q = torch.zeros(H, D, dtype=torch.float16)
    win = torch.zeros(W, D, dtype=torch.float16)
    comp = torch.zeros(4, D, dtype=torch.float16)
    tok = torch.zeros(1, D, dtype=torch.float16)
    w = torch.zeros(D, dtype=torch.float32)
    state = torch.zeros(2 + 2 * D, dtype=torch.float32)
    out = torch.zeros(H, D, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ds4a_lib.ds4a_attn_decode(q, win, win, comp, comp, None, 4, 0.125, out)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ds4a_lib.ds4a_compress_attn_decode(tok, tok, w, 128, 511, state, comp, comp, q, win, win, 0.125, out)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ds4a_lib.bind("ds4a_attn_decode", q, win, win, comp, comp, None, 4, 0.125, out)
    kidx = torch.zeros(4, 32, dtype=torch.float16)
    qi = torch.zeros(32, dtype=torch.float16)
    sel = torch.zeros(16, dtype=torch.int32)
    ws = torch.zeros(4096, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ds4a_lib.ds4a_indexer_topk_compress(qi, kidx, 19, 4, 16, sel, None, ws, tok, tok, w, state, comp, comp)


def test_wait_limit_hook_validation(ds4a_lib):
    L = ds4a_lib.lib()
    assert L.ds4a_test_set_wait_limit(-1) == ARG
    assert L.ds4a_test_set_wait_limit(20_000_000_000) == ARG
    assert L.ds4a_test_set_wait_limit(0) == 0


def _desc(ds4a_lib, **kw):
    """A ds4a_decode_layer_t of an indexer layer (H 8, D 64, W 32, ratio 4, top-16,
    d_idx 32, cap 10) on fake, aligned addresses; kw overrides fields."""
    d = ds4a_lib.DecodeLayerDesc(H=8, D=64, W=32, ratio=4, topk=16, d_idx=32, pooled_keys=0, scale=0.125, cap=10)
    for f in ("ring_k", "ring_v", "score_w", "state", "comp_k", "comp_v", "k_idx", "q", "q_idx", "out_idx", "out_n",
              "ws", "out"):
        setattr(d, f, FAKE)
    d.ws_bytes = 1 << 20
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_decode_layer_step_validation(ds4a_lib):
    """Every check runs before the first copy or launch (these return before any CUDA
    call): a missing layer, bad shapes, an indexer layer without a ratio, a missing
    array, capacity and workspace."""
    import ctypes as C
    f = ds4a_lib.lib().ds4a_decode_layer_step
    run = lambda d, pos=38: f(C.byref(d), pos, None, None, None)
    assert f(None, 0, None, None, None) == ARG
    assert run(_desc(ds4a_lib), pos=-1) == ARG
    assert run(_desc(ds4a_lib, W=0)) == ARG
    assert run(_desc(ds4a_lib, W=5000)) == ARG
    assert run(_desc(ds4a_lib, H=12)) == UNSUP
    assert run(_desc(ds4a_lib, D=96)) == UNSUP
    assert run(_desc(ds4a_lib, ratio=0)) == ARG                  # an indexer layer needs a ratio
    assert run(_desc(ds4a_lib, topk=0, pooled_keys=1)) == ARG    # pooled keys need the indexer
    assert run(_desc(ds4a_lib, pooled_keys=1)) == ARG            # ... and the token's key array
    assert run(_desc(ds4a_lib, topk=4096)) == UNSUP
    assert run(_desc(ds4a_lib, d_idx=20)) == UNSUP
    assert run(_desc(ds4a_lib, q_idx=None)) == ARG
    assert run(_desc(ds4a_lib, ring_k=FAKE + 8)) == ARG           # misaligned
    assert run(_desc(ds4a_lib, comp_v=None)) == ARG
    assert run(_desc(ds4a_lib, ws_bytes=16)) == WS
    assert run(_desc(ds4a_lib), pos=43) == CAP                   # row 10 of a 10-row capacity
    assert run(_desc(ds4a_lib, topk=0, ratio=128, cap=0), pos=128) == CAP


def test_decode_layer_struct_layout_matches_the_header(ds4a_lib, tmp_path):
    """The binding's ctypes structures have the header's field offsets and sizes
    (compiled with the host C compiler)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"ds4a_decode_layer_t": ds4a_lib.DecodeLayerDesc, "ds4a_decode_host_inputs_t": ds4a_lib.DecodeHostInputs}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "ds4a.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'printf("{cname}.{fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                                check=True).stdout.split("\n") if line)
    for cname, py in structs.items():
        assert int(got[cname]) == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert int(got[f"{cname}.{fname}"]) == getattr(py, fname).offset, f"{cname}.{fname}"


def test_host_step_binding_refuses_device_pointers_for_host_inputs(ds4a_lib):
    import torch
    d = _desc(ds4a_lib)
    with pytest.raises(ValueError, match="elements"):
        ds4a_lib.bind("ds4a_decode_layer_step", d, 38, torch.zeros(65, dtype=torch.float16))
    with pytest.raises(TypeError):
        ds4a_lib.bind("ds4a_decode_layer_step", d, 38, torch.zeros(64, dtype=torch.float32))


def test_indexer_topk_compress_keys_validation(ds4a_lib):
    f = ds4a_lib.lib().ds4a_indexer_topk_compress_keys
    # q_idx, k_idx, n_rows, d_idx, q_pos, ratio, k, out_idx, out_n, ws, ws_bytes, k_new, v_new, k_idx_tok,
    # head_dim, score_w, state, comp_k, comp_v, cap, stream
    ok = [FAKE, FAKE, 100, 64, 39, 4, 16, FAKE, None, FAKE, 1 << 20, FAKE, FAKE, FAKE, 128, FAKE, FAKE, FAKE, FAKE,
          100, None]

    def call(**kw):
        args = list(ok)
        names = ["q_idx", "k_idx", "n_rows", "d_idx", "q_pos", "ratio", "k", "out_idx", "out_n", "ws", "ws_bytes",
                 "k_new", "v_new", "k_idx_tok", "head_dim", "score_w", "state", "comp_k", "comp_v", "cap", "stream"]
        for name, v in kw.items():
            args[names.index(name)] = v
        return f(*args)
    assert call(k_idx_tok=None) == ARG          # the token's indexer key is required
    assert call(k_idx=None) == ARG              # the pooled keys are written into k_idx
    assert call(d_idx=20) == UNSUP
    assert call(k=4096) == UNSUP
    assert call(ws_bytes=8) == WS
    assert call(q_pos=403) == CAP               # completes row 100 of a 100-row capacity
    assert call(n_rows=9, q_pos=39) == CAP      # row 9 is past the 9 key rows
    assert call(k_idx_tok=FAKE + 8) == ARG      # misaligned
