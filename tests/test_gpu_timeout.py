"""The bounded device wait's give-up path, driven on the GPU without a fault.

Decode attention merges the per-head partials of its cluster's CTAs after a
bounded wait on a receive barrier; a wait that gives up records
DS4A_ERR_TIMEOUT in the device error word instead of trapping, so the context
stays usable.  The test hook ds4a_test_set_wait_limit makes CTA 0 of every
later decode attention launch also wait, after all of its partials have
arrived, on a barrier that nothing completes.  The wait must give up within
its short limit, the status must read back as DS4A_ERR_TIMEOUT, the output must
be the normal one, and the next launch without the hook must be clean.
"""
import time

import numpy as np
import pytest
import torch

from compressed_sparse_mqa_gb300 import configs, ds4a
from compressed_sparse_mqa_gb300.layer import DecodeLayer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layer", [2, 3])   # ratio 4 + indexer (attn_decode), ratio 128 (compress_attn_decode)
def test_decode_wait_gives_up_and_reports_timeout(ds4a_lib, layer):
    torch.cuda.set_device(0)
    inst = configs.decode(configs.c5_layer_params(layer, context=4096))
    a = DecodeLayer(inst)
    b = a.clone()
    assert ds4a.ds4a_last_device_error() == 0
    ref = a.step().clone()
    torch.cuda.synchronize()
    assert ds4a.ds4a_last_device_error() == 0
    try:
        ds4a.ds4a_test_set_wait_limit(100_000)          # 100 us
        t0 = time.perf_counter()
        out = b.step()
        status = ds4a.ds4a_last_device_error()          # synchronises
        dt = time.perf_counter() - t0
    finally:
        ds4a.ds4a_test_set_wait_limit(0)
    assert status == ds4a.DS4A_ERR_TIMEOUT
    assert dt < 5.0
    assert np.array_equal(out.cpu().numpy(), ref.cpu().numpy())
    # the context is usable and the next launch, without the hook, records nothing
    b.step()
    assert ds4a.ds4a_last_device_error() == 0
