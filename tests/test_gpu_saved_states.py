"""The state copies a forward saves for the backward (a training step's saved activation, like
the gate): with them the backward's dq part reads each chunk's state copy instead of scanning
the state itself.  The backward that reads them must match the fp64 oracle (bar 2e-2 of each
output's RMS) and the backward that scans -- for ragged T, an initial state, pairs cut into
parts (forward and backward), fp16/fp32 inputs, and at the training shape."""
import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, oracle_decays, rel_err, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "d_a", "d_init_state")


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    gla.load()
    yield gla, torch
    gla.set_split_parts(0)


CASES = [
    # B, T, H, input dtype, forced parts (0: automatic), seed
    (2, 256, 3, "bf16", 0, 101),
    (1, 300, 16, "bf16", 0, 102),    # ragged: a 44-token last chunk, all decay tiers
    (2, 700, 2, "bf16", 3, 103),     # pairs cut into 3 parts (forward and backward), ragged
    (1, 4000, 2, "bf16", 0, 104),    # few long sequences: the automatic cut
    (1, 384, 2, "fp16", 0, 105),
    (1, 200, 2, "fp32", 0, 106),
    (2, 1, 3, "bf16", 0, 107),       # a single token per sequence
    (2, 77, 3, "bf16", 0, 108),      # one partial chunk
]


@pytest.mark.parametrize("B,T,H,dtype,parts,seed", CASES)
def test_backward_with_saved_states(env, B, T, H, dtype, parts, seed):
    import oracle
    gla, torch = env
    td = dict(bf16=torch.bfloat16, fp16=torch.float16, fp32=torch.float32)[dtype]
    q, k, v = synth.qkv(seed, B, T, H, bf16=(dtype == "bf16"))
    dO = synth.grad_out(seed, B, T, H, bf16=(dtype == "bf16"))
    if dtype == "fp16":
        q, k, v, dO = (x.astype(np.float16).astype(np.float32) for x in (q, k, v, dO))
    a = synth.aug_balance(seed, (H, 96), 0.3)
    init = synth.init_state(seed, B, H, 0.05)
    dfin = synth.normal(seed, synth.DFIN, (B, H, 96, 192), 0.05)
    gam, gam64 = oracle_decays(H)
    gam = gam.cuda()
    qd, kd, vd, gd = (to_dev(x, td) for x in (q, k, v, dO))
    ad, idd, fd = (to_dev(x, torch.float32) for x in (a, init, dfin))
    saved = torch.empty(gla.chunk_saved_states_size(B, T, H), dtype=torch.uint8, device="cuda")
    gate = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    gla.set_split_parts(parts)
    try:
        o, fin = gla.chunk_fwd(qd, kd, vd, gam, ad, idd, gate=gate, saved_states=saved)
        g_sc = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, idd, fd, gate=gate, saved_states=saved)
        g_scan = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, idd, fd, gate=gate)
        g_sc_nogate = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, idd, fd, saved_states=saved)
        torch.cuda.synchronize()
    finally:
        gla.set_split_parts(0)
    assert gla.get_device_error() == 0
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a, init)
    ref = oracle.bwd(q, k, v, gam64, a, dO, init, dfin)
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_CHUNK
    assert rel_err(fin.cpu().numpy(), fin_ref) <= TOL_CHUNK
    errs = {}
    for name, x, y, z in zip(NAMES, g_sc, g_scan, g_sc_nogate):
        errs[name] = rel_err(x.cpu().numpy(), ref[name])
        assert errs[name] <= TOL_CHUNK, f"{name} (saved states) vs oracle: {errs[name]:.3e}"
        assert rel_err(z.cpu().numpy(), ref[name]) <= TOL_CHUNK, f"{name} (no gate)"
        # the dk, dv, d_init_state parts do not read the copies: the same kernels' results
        if name in ("dk", "dv", "d_init_state"):
            assert torch.equal(x, y), name
        else:
            assert rel_err(x.cpu().numpy(), y.cpu().numpy()) <= TOL_CHUNK, name
    print(f"saved states B={B} T={T} H={H} {dtype} parts={parts}: "
          + " ".join(f"{n} {e:.1e}" for n, e in errs.items()))


def test_saved_states_at_the_training_shape(env):
    """B=4 of the training workload's recipe (T=2048, H=16, a ~ N(0,0.02)): the forward saves
    gate and state copies, the backward reads both; every gradient against the oracle."""
    import oracle
    gla, torch = env
    x = synth.chunk_inputs("train_fwd_bwd", B=4)
    B, T, H = 4, 2048, 16
    gam, gam64 = oracle_decays(H)
    gam = gam.cuda()
    qd, kd, vd, gd = (to_dev(x[n], torch.bfloat16) for n in ("q", "k", "v", "dO"))
    ad = to_dev(x["a"], torch.float32)
    saved = torch.empty(gla.chunk_saved_states_size(B, T, H), dtype=torch.uint8, device="cuda")
    gate = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    gla.chunk_fwd(qd, kd, vd, gam, ad, gate=gate, saved_states=saved)
    g = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, gate=gate, saved_states=saved)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    ref = oracle.bwd(x["q"], x["k"], x["v"], gam64, x["a"], x["dO"])
    for name, t in zip(NAMES, g):
        e = rel_err(t.cpu().numpy(), ref[name])
        print(f"training shape, saved states: {name} {e:.2e}")
        assert e <= TOL_CHUNK, name


def test_saved_states_size_and_refusals(env):
    gla, torch = env
    B, T, H = 2, 300, 3
    n = B * H * 3  # chunks
    assert gla.chunk_saved_states_size(B, T, H) == ((n * 36864 + 255) // 256) * 256 + 4 * n
    q = torch.zeros(B, T, H, 96, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(B, T, H, 192, dtype=torch.bfloat16, device="cuda")
    gam = oracle_decays(H)[0].cuda()
    a = torch.zeros(H, 96, device="cuda")
    small = torch.empty(gla.chunk_saved_states_size(B, T, H) - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):  # the binding refuses a buffer that is too small
        gla.chunk_fwd(q, q, v, gam, a, saved_states=small)
    lib = gla.load()
    big = torch.empty(gla.chunk_saved_states_size(B, T, H) + 512, dtype=torch.uint8, device="cuda")
    o = torch.empty(B, T, H, 192, device="cuda")
    args = [q.data_ptr(), q.data_ptr(), v.data_ptr(), gla.GLA_BF16, gam.data_ptr(), a.data_ptr(),
            None, o.data_ptr(), None, None]
    tail = [None, 0, B, T, H, 96, 192, torch.cuda.current_stream().cuda_stream]
    # the C ABI: too small -> GLA_ERR_WORKSPACE, not 256-byte aligned -> GLA_ERR_ALIGNMENT
    assert lib.gla_chunk_fwd(*args, big.data_ptr(), 10, *tail) == 7
    assert lib.gla_chunk_fwd(*args, big.data_ptr() + 16, big.numel() - 16, *tail) == 3
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
