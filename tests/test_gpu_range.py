"""The fp16 operand range on the chunked paths: the tensor cores take fp16 operands, so a
legal bf16 input of magnitude >= 65504 cannot be represented there.  Each call that forms such
an operand must report GLA_ERR_RANGE in the device error word -- a status the host reads, not
a fault -- and the next call with ordinary inputs must be correct.  Large inputs that stay
inside the range must still meet the parity bar."""
import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, oracle_decays, rel_err, to_dev

pytestmark = pytest.mark.gpu

GLA_ERR_RANGE = 6
BIG = 1.0e5  # exactly representable in bf16 (1.0e5 = 0x47C3_5000 -> bf16 0x47C3 = 99840)
B, T, H = 1, 256, 2


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    gla.load()
    return gla, torch


def _inputs(seed=91):
    q, k, v = synth.qkv(seed, B, T, H)
    dO = synth.grad_out(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    return q, k, v, dO, a


def _plant(x):
    """One element set to BIG: token 127 (the last row of the first chunk, whose key/value
    decay weight is lambda^0 = 1) of head 1 (the long-memory head)."""
    x = x.copy()
    x[0, 127, 1, 5] = BIG
    return x


def _normal_call_is_correct(env):
    import oracle
    gla, torch = env
    q, k, v, dO, a = _inputs(92)
    gam, gam64 = oracle_decays(H)
    qd, kd, vd, gd = (to_dev(x, torch.bfloat16) for x in (q, k, v, dO))
    o, fin = gla.chunk_fwd(qd, kd, vd, gam.cuda(), to_dev(a, torch.float32))
    g = gla.chunk_bwd(qd, kd, vd, gam.cuda(), to_dev(a, torch.float32), gd)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a)
    ref = oracle.bwd(q, k, v, gam64, a, dO)
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_CHUNK
    assert rel_err(fin.cpu().numpy(), fin_ref) <= TOL_CHUNK
    for x, n in zip(g, ("dq", "dk", "dv", "d_a", "d_init_state")):
        assert rel_err(x.cpu().numpy(), ref[n]) <= TOL_CHUNK, n


@pytest.mark.parametrize("call,which", [("fwd", "q"), ("fwd", "k"), ("fwd", "v"),
                                        ("bwd", "q"), ("bwd", "k"), ("bwd", "v"),
                                        ("bwd", "dO")])
def test_out_of_range_bf16_input_is_reported(env, call, which):
    gla, torch = env
    q, k, v, dO, a = _inputs()
    x = dict(q=q, k=k, v=v, dO=dO)
    x[which] = _plant(x[which])
    assert synth.round_bf16(x[which])[0, 127, 1, 5] >= 65504  # a legal bf16 value, past fp16
    gam = oracle_decays(H)[0].cuda()
    qd, kd, vd, gd = (to_dev(x[n], torch.bfloat16) for n in ("q", "k", "v", "dO"))
    ad = to_dev(a, torch.float32)
    assert gla.get_device_error() == 0
    if call == "fwd":
        gla.chunk_fwd(qd, kd, vd, gam, ad)
    else:
        gla.chunk_bwd(qd, kd, vd, gam, ad, gd)
    assert gla.get_device_error() == GLA_ERR_RANGE
    _normal_call_is_correct(env)


def test_out_of_range_fp32_input_is_reported_by_the_conversion(env):
    gla, torch = env
    q, k, v, dO, a = _inputs()
    gam = oracle_decays(H)[0].cuda()
    v = _plant(v)
    gla.chunk_fwd(to_dev(q, torch.float32), to_dev(k, torch.float32), to_dev(v, torch.float32),
                  gam, to_dev(a, torch.float32))
    assert gla.get_device_error() == GLA_ERR_RANGE
    _normal_call_is_correct(env)


@pytest.mark.parametrize("which", ["state", "adjoint"])
def test_out_of_range_input_is_reported_by_the_slice_sums(env, which):
    """The segment passes (here through the slice sums, which run them alone)."""
    gla, torch = env
    q, k, v, dO, a = _inputs()
    gam = oracle_decays(H)[0].cuda()
    if which == "state":
        gla.chunk_state_sum(to_dev(k, torch.bfloat16), to_dev(_plant(v), torch.bfloat16), gam)
    else:
        gla.chunk_adjoint_sum(to_dev(q, torch.bfloat16), to_dev(_plant(dO), torch.bfloat16), gam)
    assert gla.get_device_error() == GLA_ERR_RANGE
    _normal_call_is_correct(env)


def test_out_of_range_input_is_reported_on_a_cut_pair(env):
    """A long sequence whose pairs are cut into parts: its segment passes and the main kernel
    run; the planted value (in a part the passes sum) is reported."""
    gla, torch = env
    Tl = 4000
    assert gla.split_plan(1, Tl, H, False, 152)[1] > 1
    q, k, v = synth.qkv(93, 1, Tl, H)
    a = synth.aug_balance(93, (H, 96), 0.1)
    v = v.copy()
    v[0, 127, 1, 5] = BIG
    gam = oracle_decays(H)[0].cuda()
    gla.chunk_fwd(to_dev(q, torch.bfloat16), to_dev(k, torch.bfloat16),
                  to_dev(v, torch.bfloat16), gam, to_dev(a, torch.float32))
    assert gla.get_device_error() == GLA_ERR_RANGE
    _normal_call_is_correct(env)


def test_large_in_range_values_meet_the_bar(env):
    """v scaled by 256 on the long-memory heads (|v| up to ~1.2e3, the states and scores of
    those heads ~1e4): inside fp16's range, so no error, and the forward and backward still
    match the oracle at the training length."""
    import oracle
    gla, torch = env
    Bn, Tn, Hn, seed = 2, 2048, 16, 94
    q, k, v = synth.qkv(seed, Bn, Tn, Hn)
    dO = synth.grad_out(seed, Bn, Tn, Hn)
    v = synth.round_bf16(v * np.where(np.arange(Hn) >= Hn // 2, 256.0, 1.0)[None, None, :, None]
                         .astype(np.float32))
    a = synth.aug_balance(seed, (Hn, 96), 0.02)
    gam, gam64 = oracle_decays(Hn)
    qd, kd, vd, gd = (to_dev(x, torch.bfloat16) for x in (q, k, v, dO))
    ad = to_dev(a, torch.float32)
    o, fin = gla.chunk_fwd(qd, kd, vd, gam.cuda(), ad)
    g = gla.chunk_bwd(qd, kd, vd, gam.cuda(), ad, gd)
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    o_ref, fin_ref = oracle.fwd(q, k, v, gam64, a)
    ref = oracle.bwd(q, k, v, gam64, a, dO)
    errs = dict(o=rel_err(o.cpu().numpy(), o_ref), final=rel_err(fin.cpu().numpy(), fin_ref))
    for x, n in zip(g, ("dq", "dk", "dv", "d_a", "d_init_state")):
        errs[n] = rel_err(x.cpu().numpy(), ref[n])
    print("large in-range v: " + " ".join(f"{n} {e:.1e}" for n, e in errs.items()))
    for n, e in errs.items():
        assert e <= TOL_CHUNK, f"{n}: {e:.3e}"
