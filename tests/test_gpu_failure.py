"""The failure path of the kernels' bounded waits, on the GPU and without a fault: a wait
that nothing completes gives up after the configured limit, the device error word reads
GLA_ERR_TIMEOUT on the host, and the context keeps working."""
import time

import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, rel_err, to_dev, oracle_decays

pytestmark = pytest.mark.gpu

GLA_ERR_TIMEOUT = 5


def test_wait_gives_up_and_reports_timeout():
    import torch
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    gla.load()
    assert gla.get_device_error() == 0
    try:
        gla.set_wait_timeout_ns(2_000_000)  # 2 ms
        t0 = time.perf_counter()
        gla.wait_probe()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert gla.get_device_error() == GLA_ERR_TIMEOUT
        assert gla.get_device_error() == 0  # read and cleared
        assert dt < 5.0
    finally:
        gla.set_wait_timeout_ns(0)  # back to the default limit
    # the context is still usable: a forward call after the timeout is correct
    import oracle
    B, T, H = 1, 256, 2
    q, k, v = synth.qkv(91, B, T, H)
    a = synth.aug_balance(91, (H, 96), 0.1)
    o, _ = gla.chunk_fwd(to_dev(q, torch.bfloat16), to_dev(k, torch.bfloat16),
                         to_dev(v, torch.bfloat16), oracle_decays(H)[0].cuda(),
                         to_dev(a, torch.float32))
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    o_ref, _ = oracle.fwd(q, k, v, oracle_decays(H)[1], a)
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_CHUNK
