"""First calls into the library from many host threads at once.

The library looks up per-device constants (the device error word's address, the
SM count, the scratch array of the allocation-free indexer) on the first call
that needs them.  This test starts a fresh process, so that nothing is set up
yet, and makes sixteen threads issue their first calls together (ctypes drops the
GIL for the duration of a foreign call, so they overlap in the C code).  Every
call is enqueued on one shared stream, so the kernels themselves run one after
another; each thread's kept rows must equal those of the same call made alone.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent(r"""
    import ctypes, sys, threading
    import numpy as np, torch
    sys.path.insert(0, ROOT)
    from compressed_sparse_mqa_gb300 import ds4a
    torch.cuda.set_device(0)
    torch.zeros(1, device="cuda")            # the CUDA context exists; the library has made no call yet
    lib = ctypes.CDLL(ds4a.LIB_PATH)
    P, I, LL, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
    lib.ds4a_indexer_topk_noalloc.argtypes = [P, P, LL, I, LL, I, I, P, P, P]
    lib.ds4a_indexer_topk.argtypes = [P, I, P, LL, I, LL, I, I, P, P, P, SZ, P]
    lib.ds4a_indexer_workspace_bytes.argtypes = [I, LL, I]
    lib.ds4a_indexer_workspace_bytes.restype = SZ
    lib.ds4a_last_device_error.argtypes = [P]
    N, n_rows, d, k, q_pos = 16, 4096, 64, 256, 4 * 4096
    rng = np.random.default_rng(1)
    kidx = torch.from_numpy(rng.standard_normal((n_rows, d)).astype(np.float16)).cuda()
    qs = [torch.from_numpy(rng.standard_normal(d).astype(np.float16)).cuda() for _ in range(N)]
    outs_a = [torch.full((k,), -5, dtype=torch.int32, device="cuda") for _ in range(N)]
    outs_b = [torch.full((k,), -5, dtype=torch.int32, device="cuda") for _ in range(N)]
    nb = lib.ds4a_indexer_workspace_bytes(1, n_rows, k)
    wss = [torch.zeros(nb, dtype=torch.uint8, device="cuda") for _ in range(N)]
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    torch.cuda.synchronize()
    go = threading.Barrier(N)
    rcs = [None] * N

    def worker(i):
        go.wait()
        r1 = lib.ds4a_indexer_topk_noalloc(qs[i].data_ptr(), kidx.data_ptr(), n_rows, d, q_pos, 4, k,
                                           outs_a[i].data_ptr(), None, sh)
        r2 = lib.ds4a_indexer_topk(qs[i].data_ptr(), 1, kidx.data_ptr(), n_rows, d, q_pos, 4, k,
                                   outs_b[i].data_ptr(), None, wss[i].data_ptr(), nb, sh)
        rcs[i] = (r1, r2)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(N)]
    for t in ts: t.start()
    for t in ts: t.join()
    torch.cuda.synchronize()
    assert all(rc == (0, 0) for rc in rcs), rcs
    assert lib.ds4a_last_device_error(None) == 0
    for i in range(N):
        ref = torch.full((k,), -5, dtype=torch.int32, device="cuda")
        assert lib.ds4a_indexer_topk(qs[i].data_ptr(), 1, kidx.data_ptr(), n_rows, d, q_pos, 4, k,
                                     ref.data_ptr(), None, wss[i].data_ptr(), nb, None) == 0
        torch.cuda.synchronize()
        assert torch.equal(outs_a[i], ref) and torch.equal(outs_b[i], ref), i
    print("threads ok")
""")


def test_first_calls_from_many_threads(ds4a_lib):
    code = "ROOT = " + repr(ROOT) + "\n" + SCRIPT
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout
