"""The indexer entry point that allocates nothing (ds4a_indexer_topk_noalloc).

Some callers cannot hand the library a workspace -- plugin or callback hosts
whose enqueue step may not allocate device memory, or programs under a fixed
memory budget -- so the library also offers a one-query indexer whose scratch is
a static device array inside the library.  This test calls it through the C ABI
and checks that, on two calls in a row, it keeps exactly the rows (and counts)
that the workspace entry point ds4a_indexer_topk keeps for the same inputs.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity import check_sel

pytestmark = pytest.mark.gpu

DS4A_OK, DS4A_ERR_WORKSPACE = 0, 6
MAX_ROWS = 65536


def _noalloc(lib):
    f = lib.ds4a_indexer_topk_noalloc
    P, I, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    f.argtypes = [P, P, LL, I, LL, I, I, P, P, P]
    f.restype = I
    return f


def _with_workspace(lib):
    f = lib.ds4a_indexer_topk
    P, I, LL, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
    f.argtypes = [P, I, P, LL, I, LL, I, I, P, P, P, SZ, P]
    f.restype = I
    lib.ds4a_indexer_workspace_bytes.argtypes = [I, LL, I]
    lib.ds4a_indexer_workspace_bytes.restype = SZ
    return f


# the last case passes more rows than the scratch holds, of which the query sees only
# floor((q_pos + 1) / 4) = 50001: the limit counts visible rows
@pytest.mark.parametrize("n_rows,d_idx,k,q_pos", [(8192, 128, 512, 32768), (20000, 64, 100, 4 * 20000 + 1),
                                                  (300, 32, 512, 4 * 300 + 3), (70000, 64, 512, 200006)])
def test_noalloc_indexer_matches_workspace_indexer(ds4a_lib, n_rows, d_idx, k, q_pos):
    assert torch.cuda.is_available()
    lib = ctypes.CDLL(ds4a_lib.LIB_PATH)
    noalloc, with_ws = _noalloc(lib), _with_workspace(lib)
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(n_rows)
    for call in range(2):   # two calls in a row, fresh inputs each time
        kidx = torch.from_numpy(rng.standard_normal((n_rows, d_idx)).astype(np.float16)).cuda()
        q = torch.from_numpy(rng.standard_normal(d_idx).astype(np.float16)).cuda()
        ref_idx = torch.full((k,), -7, dtype=torch.int32, device="cuda")
        ref_n = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = torch.zeros(lib.ds4a_indexer_workspace_bytes(1, n_rows, k), dtype=torch.uint8, device="cuda")
        assert with_ws(q.data_ptr(), 1, kidx.data_ptr(), n_rows, d_idx, q_pos, 4, k, ref_idx.data_ptr(),
                       ref_n.data_ptr(), ws.data_ptr(), ws.numel(), stream) == DS4A_OK
        got_idx = torch.full((k,), -9, dtype=torch.int32, device="cuda")
        got_n = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert noalloc(q.data_ptr(), kidx.data_ptr(), n_rows, d_idx, q_pos, 4, k, got_idx.data_ptr(),
                       got_n.data_ptr(), stream) == DS4A_OK
        torch.cuda.synchronize()
        n_vis = min(n_rows, (q_pos + 1) // 4)
        assert int(got_n.item()) == int(ref_n.item()) == min(k, n_vis)
        # kept rows are integers: bit-exact
        assert torch.equal(got_idx, ref_idx), f"call {call}: rows differ"
        if call == 1:
            # and against the oracle: the same rows up to near-ties of the k-th score
            q_h, k_h = q.cpu().numpy(), kidx[:n_vis].cpu().numpy()
            scores = oracle.index_scores(q_h, k_h)
            check_sel(got_idx.cpu().numpy(), oracle.topk(scores, k), scores, k, "noalloc vs oracle")
    assert ds4a_lib.ds4a_last_device_error() == 0


def test_noalloc_indexer_rejects_rows_beyond_its_scratch(ds4a_lib):
    lib = ctypes.CDLL(ds4a_lib.LIB_PATH)
    noalloc = _noalloc(lib)
    n_rows = MAX_ROWS + 1
    kidx = torch.zeros(n_rows, 128, dtype=torch.float16, device="cuda")
    q = torch.zeros(128, dtype=torch.float16, device="cuda")
    out = torch.full((512,), -3, dtype=torch.int32, device="cuda")
    rc = noalloc(q.data_ptr(), kidx.data_ptr(), n_rows, 128, 4 * n_rows, 4, 512, out.data_ptr(), None,
                 torch.cuda.current_stream().cuda_stream)
    assert rc == DS4A_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (out == -3).all()   # nothing was enqueued
