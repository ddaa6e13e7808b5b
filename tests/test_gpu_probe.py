"""The gather-rate measurement call (ds4a_probe_gather): it runs on valid row lists
without recording anything, and skips and records rows outside its table."""
import pytest
import torch

from compressed_sparse_mqa_gb300 import ds4a

pytestmark = pytest.mark.gpu


def test_probe_gather_runs_and_flags_bad_rows(ds4a_lib):
    torch.cuda.set_device(0)
    table = torch.randn(1000, 128, device="cuda").half()
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.randint(0, 1000, (5000,), dtype=torch.int32, device="cuda")
    ds4a.ds4a_probe_gather(table, idx, sink)
    assert ds4a.ds4a_last_device_error() == 0
    idx[17] = 1000
    ds4a.ds4a_probe_gather(table, idx, sink)
    assert ds4a.ds4a_last_device_error() == ds4a.DS4A_ERR_DEVICE_INDEX
    assert ds4a.ds4a_last_device_error() == 0
