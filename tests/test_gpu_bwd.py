"""GPU parity of gla_chunk_bwd against the fp64 oracle (bar: 2e-2 of each output's RMS)."""
import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, as_dtype_values, rel_err, to_dev, oracle_decays

pytestmark = pytest.mark.gpu

TDT = {"bf16": "bfloat16", "fp16": "float16", "fp32": "float32"}
NAMES = ("dq", "dk", "dv", "d_a", "d_init_state")


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    gla.load()
    return gla, torch


def run_bwd(env, q, k, v, a, dO, init, dfin, H, dtype):
    import oracle
    gla, torch = env
    td = getattr(torch, TDT[dtype])
    q, k, v, dO = (as_dtype_values(x, dtype) for x in (q, k, v, dO))
    gam = oracle_decays(H)[0]
    gam64 = oracle_decays(H)[1]
    f32 = lambda x: None if x is None else to_dev(x, torch.float32)
    dq, dk, dv, da, dinit = gla.chunk_bwd(to_dev(q, td), to_dev(k, td), to_dev(v, td), gam.cuda(),
                                          f32(a), to_dev(dO, td), f32(init), f32(dfin))
    torch.cuda.synchronize()
    assert gla.get_device_error() == 0
    got = dict(dq=dq, dk=dk, dv=dv, d_a=da, d_init_state=dinit)
    got = {n: x.cpu().numpy() for n, x in got.items()}
    ref = oracle.bwd(q, k, v, gam64, a, dO, init, dfin)
    return got, ref


CASES = [
    # B, T, H, dtype, init std, d_final std, a std, seed
    (1, 128, 1, "bf16", 0.0, 0.0, 0.1, 31),
    (2, 384, 5, "bf16", 0.05, 0.05, 0.1, 32),
    (1, 256, 2, "fp16", 0.05, 0.02, 0.1, 33),
    (3, 640, 16, "bf16", 0.02, 0.01, 0.02, 34),
    # ragged: the last chunk (the reverse scans' first) holds T mod 128 tokens
    (2, 1, 3, "bf16", 0.05, 0.05, 0.1, 35),
    (2, 77, 3, "bf16", 0.05, 0.05, 0.1, 36),
    (2, 200, 16, "bf16", 0.02, 0.05, 0.02, 37),
    (1, 300, 2, "fp32", 0.05, 0.05, 0.1, 38),
    (3, 511, 5, "fp16", 0.02, 0.02, 0.1, 39),
]


@pytest.mark.parametrize("B,T,H,dtype,init_std,dfin_std,a_std,seed", CASES)
def test_bwd_small(env, B, T, H, dtype, init_std, dfin_std, a_std, seed):
    q, k, v = synth.qkv(seed, B, T, H, bf16=False)
    dO = synth.grad_out(seed, B, T, H, bf16=False)
    a = synth.aug_balance(seed, (H, 96), a_std)
    init = synth.init_state(seed, B, H, init_std) if init_std > 0 else None
    dfin = synth.normal(seed, synth.DFIN, (B, H, 96, 192), dfin_std) if dfin_std > 0 else None
    got, ref = run_bwd(env, q, k, v, a, dO, init, dfin, H, dtype)
    errs = {n: rel_err(got[n], ref[n]) for n in NAMES}
    print(f"bwd B={B} T={T} H={H} {dtype}: " + " ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL_CHUNK for e in errs.values()), errs


def test_bwd_tiny_fp32_workload(env):
    x = synth.chunk_inputs("tiny_fp32")
    got, ref = run_bwd(env, x["q"], x["k"], x["v"], x["a"], x["dO"], None, None, x["cfg"]["H"],
                       "fp32")
    errs = {n: rel_err(got[n], ref[n]) for n in NAMES}
    print("bwd tiny fp32: " + " ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL_CHUNK for e in errs.values()), errs


def test_bwd_training_workload(env):
    """Training shape: B=32, T=2048, H=16, bf16, a ~ N(0, 0.02), dO ~ N(0, 1): every
    gradient (dq, dk, dv, d_aug, d_init_state) against the oracle."""
    x = synth.chunk_inputs("train_fwd_bwd")
    got, ref = run_bwd(env, x["q"], x["k"], x["v"], x["a"], x["dO"], None, None, x["cfg"]["H"],
                       "bf16")
    errs = {n: rel_err(got[n], ref[n]) for n in NAMES}
    print("bwd train: " + " ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL_CHUNK for e in errs.values()), errs
