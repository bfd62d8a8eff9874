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


@pytest.mark.parametrize("case,step", [("fwd", 0), ("fwd", 2), ("bwd", 0), ("bwd", 3),
                                       ("cut_fwd", 1), ("cut_bwd", 1),
                                       ("overlap_fwd", 0), ("overlap_bwd", 0)])
def test_chunk_kernel_waits_give_up_and_the_next_call_is_correct(case, step):
    """The chunk kernels' own waits run out: with gla_set_stall_step the tensor-core issuer of
    every CTA waits, at chunk step `step`, on a barrier that completes only after its loop, so
    its bounded wait (2 ms here) gives up and raises the CTA's abort flag.  Every role then
    leaves its loop on one path per warp (the epilogue warps vote), drains its copies and
    MMAs and frees its tensor memory.  The host reads GLA_ERR_TIMEOUT; with the diagnostic off
    the next forward and backward are correct.  The cut_* cases cut every pair (the segment
    passes run first); the overlap_* cases have a full wave of whole pairs and 8 cut ones, so
    the passes and the chunked kernel are chained as programmatic dependent launches: the
    passes' own waits give up, they complete, and the parts' griddepcontrol.wait returns."""
    import torch
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    gla.load()
    import oracle
    B, H = 1, 2
    T = 4000 if case.startswith("cut") else 640  # 4000: the pairs are cut into parts
    if case.startswith("overlap"):
        if torch.cuda.get_device_properties(0).multi_processor_count != 152:
            pytest.skip("the layout of this case assumes 152 SMs")
        B, H, T = 10, 16, 256  # 160 pairs: 152 whole, the last 8 cut in 2 (forced)
    q, k, v = synth.qkv(95, B, T, H)
    dO = synth.grad_out(95, B, T, H)
    a = synth.aug_balance(95, (H, 96), 0.1)
    gam, gam64 = oracle_decays(H)
    qd, kd, vd, gd = (to_dev(x, torch.bfloat16) for x in (q, k, v, dO))
    ad = to_dev(a, torch.float32)
    assert gla.get_device_error() == 0
    try:
        if case.startswith("overlap"):
            gla.set_split_parts(2)
            assert gla.split_plan(B, T, H, case.endswith("bwd"), 152) == (152, 2)
        gla.set_wait_timeout_ns(2_000_000)
        gla.set_stall_step(step)
        t0 = time.perf_counter()
        if case.endswith("fwd"):
            gla.chunk_fwd(qd, kd, vd, gam.cuda(), ad)
        else:
            gla.chunk_bwd(qd, kd, vd, gam.cuda(), ad, gd)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert gla.get_device_error() == GLA_ERR_TIMEOUT
        assert dt < 5.0
    finally:
        gla.set_stall_step(-1)
        gla.set_wait_timeout_ns(0)
        gla.set_split_parts(0)
    o, fin = gla.chunk_fwd(qd, kd, vd, gam.cuda(), ad)
    g = gla.chunk_bwd(qd, kd, vd, gam.cuda(), ad, gd)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a)
    ref = oracle.bwd(q, k, v, gam64, a, dO)
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_CHUNK
    assert rel_err(fin.cpu().numpy(), fin_ref) <= TOL_CHUNK
    for x, n in zip(g, ("dq", "dk", "dv", "d_a", "d_init_state")):
        assert rel_err(x.cpu().numpy(), ref[n]) <= TOL_CHUNK, n
