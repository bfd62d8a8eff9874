"""The gate sigmoid(q.(a*k)) saved by the forward for the backward (a training step's saved
activation): the forward writes it (checked against the oracle's gate), and the backward
that reads it matches the fp64 oracle (bar 2e-2 of each output's RMS) and the backward that
recomputes it -- for ragged T, pairs cut into parts, fp16/fp32 inputs and the no-workspace
call."""
import ctypes

import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, rel_err, to_dev, oracle_decays

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "d_a", "d_init_state")
# sigmoid of an fp32 dot product of the bf16/fp16 values against fp64; fp32 inputs go through
# the fp16 copies the library makes of them, so q and k carry 2^-11 relative rounding each:
# |dz| <= 2^-10 sum|a q k| (~1 here) and sigmoid' <= 1/4
GATE_TOL = dict(bf16=1e-5, fp16=1e-5, fp32=5e-4)


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
    (2, 256, 3, "bf16", 0, 71),
    (1, 300, 16, "bf16", 0, 72),    # ragged: a 44-token last chunk
    (2, 700, 2, "bf16", 3, 73),     # pairs cut into 3 parts, ragged
    (1, 384, 2, "fp16", 0, 74),
    (1, 200, 2, "fp32", 0, 75),
    (2, 1, 3, "bf16", 0, 78),       # a single token per sequence
    (2, 77, 3, "bf16", 0, 79),      # one partial chunk
]


@pytest.mark.parametrize("B,T,H,dtype,parts,seed", CASES)
def test_saved_gate_forward_and_backward(env, B, T, H, dtype, parts, seed):
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
    gam = oracle_decays(H)[0].cuda()
    gam64 = oracle_decays(H)[1]
    qd, kd, vd, gd = (to_dev(x, td) for x in (q, k, v, dO))
    ad, idd, fd = (to_dev(x, torch.float32) for x in (a, init, dfin))
    gla.set_split_parts(parts)
    try:
        gate = torch.full((B, H, T), float("nan"), dtype=torch.float32, device="cuda")
        o, fin = gla.chunk_fwd(qd, kd, vd, gam, ad, idd, gate=gate)
        g_saved = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, idd, fd, gate=gate)
        g_rec = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, idd, fd)
        torch.cuda.synchronize()
        assert gla.get_device_error() == 0
    finally:
        gla.set_split_parts(0)
    gate_ref = oracle.gate(q, k, a)
    eg = float(np.abs(gate.cpu().numpy() - gate_ref.transpose(0, 2, 1)).max())
    o_ref, _ = oracle.fwd(q, k, v, gam64, a, init)
    ref = oracle.bwd(q, k, v, gam64, a, dO, init, dfin)
    errs = {n: rel_err(x.cpu().numpy(), ref[n]) for n, x in zip(NAMES, g_saved)}
    vs_rec = {n: rel_err(x.cpu().numpy(), y.cpu().numpy()) for n, x, y in zip(NAMES, g_saved, g_rec)}
    print(f"gate B={B} T={T} H={H} {dtype} parts={parts}: gate {eg:.1e} | " +
          " ".join(f"{n} {e:.2e}" for n, e in errs.items()) +
          " | vs recomputed " + " ".join(f"{n} {e:.1e}" for n, e in vs_rec.items()))
    assert eg <= GATE_TOL[dtype]
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_CHUNK
    assert all(e <= TOL_CHUNK for e in errs.values()), errs
    # the two backwards differ only by the rounding of the gate's dot product
    assert all(e <= 1e-3 for e in vs_rec.values()), vs_rec


def test_backward_follows_the_gate_it_is_given(env):
    """Given the gate of another balance a2, the backward's outputs are the oracle's for a2
    where only the gate depends on a (dk, dv away from the self-augmentation term are not a
    test of that); checked on d_aug = sum r (q*k), r = sigmoid'(z) (dO.v): with the gate of
    a2 = 0 (every value 1/2) it is sum (dO.v)/4 (q*k) whatever a is."""
    gla, torch = env
    B, T, H, seed = 1, 256, 2, 76
    q, k, v = synth.qkv(seed, B, T, H)
    dO = synth.grad_out(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.3)
    qd, kd, vd, gd = (to_dev(x, torch.bfloat16) for x in (q, k, v, dO))
    gate = torch.full((B, H, T), 0.5, dtype=torch.float32, device="cuda")
    _, _, _, d_aug, _ = gla.chunk_bwd(qd, kd, vd, oracle_decays(H)[0].cuda(),
                                      to_dev(a, torch.float32), gd, gate=gate)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    dov = np.einsum("bthc,bthc->bth", dO.astype(np.float64), v.astype(np.float64))
    expect = np.einsum("bth,bthc->hc", 0.25 * dov, q.astype(np.float64) * k.astype(np.float64))
    e = rel_err(d_aug.cpu().numpy(), expect)
    print(f"d_aug with the gate of a = 0: {e:.2e}")
    assert e <= TOL_CHUNK


def test_no_workspace_backward_reads_the_gate(env):
    gla, torch = env
    B, T, H, seed = 2, 384, 3, 77
    q, k, v = synth.qkv(seed, B, T, H)
    dO = synth.grad_out(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.3)
    qd, kd, vd, gd = (to_dev(x, torch.bfloat16) for x in (q, k, v, dO))
    ad = to_dev(a, torch.float32)
    gam = oracle_decays(H)[0].cuda()
    gate = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    gla.chunk_fwd(qd, kd, vd, gam, ad, gate=gate)
    gla.set_split_parts(1)  # the no-workspace call never cuts pairs: compare like with like
    try:
        ref = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, gate=gate, want_d_init_state=False)
    finally:
        gla.set_split_parts(0)
    lib = gla.load()
    fn = lib.gla_chunk_bwd_noalloc
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] + [ctypes.c_void_p] * 11 + \
        [ctypes.c_int] * 5 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    f32 = dict(dtype=torch.float32, device="cuda")
    out = [torch.empty((B, T, H, 96), **f32), torch.empty((B, T, H, 96), **f32),
           torch.empty((B, T, H, 192), **f32), torch.empty((H, 96), **f32)]
    rc = fn(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), gla.GLA_BF16, gam.data_ptr(),
            ad.data_ptr(), None, gd.data_ptr(), None, gate.data_ptr(),
            *[x.data_ptr() for x in out], None, B, T, H, 96, 192,
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, gla.status_string(rc)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    for name, x, r in zip(NAMES, out, ref):
        assert torch.equal(x, r), f"{name} differs between the no-workspace and workspace calls"


def test_saved_gate_at_the_training_shape(env):
    """B=8, T=2048, H=16 (one training-shape layer): the backward that reads the forward's gate
    against the one that recomputes it (they differ only by the rounding of the gate's dot
    product), and the gate against the oracle's on sampled rows."""
    import oracle
    gla, torch = env
    B, T, H, seed = 8, 2048, 16, 80
    q, k, v = synth.qkv(seed, B, T, H)
    dO = synth.grad_out(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.02)
    qd, kd, vd, gd = (to_dev(x, torch.bfloat16) for x in (q, k, v, dO))
    ad = to_dev(a, torch.float32)
    gam = oracle_decays(H)[0].cuda()
    gate = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    gla.chunk_fwd(qd, kd, vd, gam, ad, gate=gate)
    g_saved = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, gate=gate)
    g_rec = gla.chunk_bwd(qd, kd, vd, gam, ad, gd)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    vs_rec = {n: rel_err(x.cpu().numpy(), y.cpu().numpy()) for n, x, y in zip(NAMES, g_saved, g_rec)}
    rows = np.random.default_rng(seed).integers(0, T, 64)
    g_ref = oracle.gate(q[:, rows], k[:, rows], a)  # [B, 64, H]
    eg = float(np.abs(gate.cpu().numpy()[:, :, rows] - g_ref.transpose(0, 2, 1)).max())
    print(f"saved gate B={B} T={T} H={H}: gate {eg:.1e} | vs recomputed " +
          " ".join(f"{n} {e:.1e}" for n, e in vs_rec.items()))
    assert eg <= GATE_TOL["bf16"]
    assert all(e <= 1e-3 for e in vs_rec.values()), vs_rec
