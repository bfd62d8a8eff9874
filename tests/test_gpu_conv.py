"""GPU parity of the causal depth-wise conv + SiLU (forward, gradient, decode step) against
the fp64 oracle: fp32 arithmetic, bar 1e-4 of the RMS of each output."""
import numpy as np
import pytest

import synth
from _util import TOL_DECODE, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    gla.load()
    return gla, torch


def _inputs(seed, B, T, D, bf16, with_init, with_bias):
    x = synth.normal(seed, synth.V, (B, T, D), 1.0)
    if bf16:
        x = synth.round_bf16(x)
    w = synth.normal(seed, synth.A, (D, 4), 0.5)
    b = synth.normal(seed, synth.DFIN, (D,), 0.1) if with_bias else None
    init = synth.normal(seed, synth.INIT, (B, 3, D), 1.0) if with_init else None
    dy = synth.normal(seed, synth.DO, (B, T, D), 1.0)
    return x, w, b, init, dy


@pytest.mark.parametrize("B,T,D,bf16,with_init,with_bias,seed", [
    (2, 67, 96, True, True, True, 81),       # forward: two full 32-token tiles and a ragged one
    (2, 259, 96, True, True, True, 88),      # backward: two full 128-token tiles, 3 tokens left
    (1, 2, 8, False, True, True, 82),        # shorter than the state
    (3, 200, 3072, True, False, False, 83),  # the model width, no state, no bias
    (4, 2048, 3072, True, True, True, 84),   # training shape (B=4 of 32)
    (2, 130, 1032, True, False, True, 86),   # a last channel block of 8 (staged forward)
    (2, 70, 1028, True, True, True, 85),     # bf16 rows not 16-byte multiples: register forward
    (2, 100, 200, False, True, False, 87),   # fp32 x, staged forward
])
def test_conv_matches_oracle(env, B, T, D, bf16, with_init, with_bias, seed):
    import oracle
    gla, torch = env
    x, w, b, init, dy = _inputs(seed, B, T, D, bf16, with_init, with_bias)
    xd = to_dev(x, torch.bfloat16 if bf16 else torch.float32)
    wd, dyd = to_dev(w, torch.float32), to_dev(dy, torch.float32)
    bd = None if b is None else to_dev(b, torch.float32)
    idd = None if init is None else to_dev(init, torch.float32)
    y, fin = gla.conv_fwd(xd, wd, bd, idd)
    dx, dinit, dw, db = gla.conv_bwd(xd, wd, dyd, bd, idd)
    torch.cuda.synchronize()
    y_ref, fin_ref = oracle.conv_fwd(x, w, b, init)
    dx_ref, di_ref, dw_ref, db_ref = oracle.conv_bwd(x, w, dy, b, init)
    errs = dict(y=rel_err(y.cpu().numpy(), y_ref), dx=rel_err(dx.cpu().numpy(), dx_ref),
                d_init=rel_err(dinit.cpu().numpy(), di_ref), d_weight=rel_err(dw.cpu().numpy(), dw_ref),
                d_bias=rel_err(db.cpu().numpy(), db_ref))
    print(f"conv B={B} T={T} D={D}: " + " ".join(f"{k} {v:.1e}" for k, v in errs.items()))
    assert np.array_equal(fin.cpu().numpy(), fin_ref.astype(np.float32))  # a copy of inputs
    for k, e in errs.items():
        assert e <= TOL_DECODE, k


def test_conv_decode_steps_equal_forward(env):
    import oracle
    gla, torch = env
    N, T, D = 5, 7, 3072
    x, w, b, init, _ = _inputs(85, N, T, D, False, True, True)
    st = to_dev(init, torch.float32)
    wd, bd = to_dev(w, torch.float32), to_dev(b, torch.float32)
    ys = [gla.conv_decode_step(st, to_dev(np.ascontiguousarray(x[:, t]), torch.float32), wd, bd)
          for t in range(T)]
    torch.cuda.synchronize()
    y = np.stack([v.cpu().numpy() for v in ys], 1)
    y_ref, fin_ref = oracle.conv_fwd(x, w, b, init)
    assert rel_err(y, y_ref) <= TOL_DECODE
    assert np.array_equal(st.cpu().numpy(), fin_ref.astype(np.float32))


def test_conv_gradients_are_deterministic(env):
    gla, torch = env
    x, w, b, init, dy = _inputs(86, 4, 512, 3072, True, True, True)
    args = (to_dev(x, torch.bfloat16), to_dev(w, torch.float32), to_dev(dy, torch.float32),
            to_dev(b, torch.float32), to_dev(init, torch.float32))
    r1, r2 = gla.conv_bwd(*args), gla.conv_bwd(*args)
    assert all(torch.equal(a, c) for a, c in zip(r1, r2))
