"""GPU parity of the output epilogue (Head RMSNorm per decay tier, SiLU(g) gate) and its
gradient against the fp64 oracle: fp32 arithmetic, bar 1e-4 of the RMS of each output."""
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


def _inputs(seed, N, H, n_tiers, g_bf16):
    o = synth.normal(seed, synth.V, (N, H, 192), 1.0)
    g = synth.normal(seed, synth.Q, (N, H, 192), 1.5)
    if g_bf16:
        g = synth.round_bf16(g)
    w = 1.0 + synth.normal(seed, synth.A, (n_tiers, 192), 0.2)
    dy = synth.normal(seed, synth.DO, (N, H, 192), 1.0)
    return o, g, w, dy


@pytest.mark.parametrize("N,H,n_tiers,g_bf16,eps,seed", [
    (37, 16, 4, True, 1e-6, 71),     # ragged token count, 4 tiers of 4 heads
    (64, 16, 16, False, 1e-5, 72),   # one head per tier, fp32 gate
    (9, 5, 5, True, 1e-6, 73),       # odd head count
    (50, 6, 1, False, 0.0, 74),      # one shared norm, eps = 0
    (8 * 2048, 16, 4, True, 1e-6, 75),  # one training-shape layer (B=8, T=2048)
    (4097, 5, 5, True, 1e-6, 77),    # odd row count over two grid passes: the two halves of a
                                     # warp run different numbers of rows
])
def test_head_norm_gate_matches_oracle(env, N, H, n_tiers, g_bf16, eps, seed):
    import oracle
    gla, torch = env
    o, g, w, dy = _inputs(seed, N, H, n_tiers, g_bf16)
    od, wd, dyd = (to_dev(x, torch.float32) for x in (o, w, dy))
    gd = to_dev(g, torch.bfloat16 if g_bf16 else torch.float32)
    y, rstd = gla.head_norm_gate(od, gd, wd, n_tiers, eps, want_rstd=True)
    d_o, dg, d_w = gla.head_norm_gate_bwd(dyd, od, gd, wd, n_tiers, eps)
    torch.cuda.synchronize()
    y_ref, r_ref = oracle.head_norm_gate(o, g, w, n_tiers, eps)
    do_ref, dg_ref, dw_ref = oracle.head_norm_gate_bwd(dy, o, g, w, n_tiers, eps)
    errs = dict(y=rel_err(y.cpu().numpy(), y_ref), rstd=rel_err(rstd.cpu().numpy(), r_ref),
                d_o=rel_err(d_o.cpu().numpy(), do_ref), dg=rel_err(dg.cpu().numpy(), dg_ref),
                d_weight=rel_err(d_w.cpu().numpy(), dw_ref))
    print(f"head norm N={N} H={H} tiers={n_tiers}: " +
          " ".join(f"{k} {v:.1e}" for k, v in errs.items()))
    for k, e in errs.items():
        assert e <= TOL_DECODE, k


def test_head_norm_weight_gradient_is_deterministic(env):
    gla, torch = env
    o, g, w, dy = _inputs(76, 4096, 16, 4, True)
    args = [to_dev(o, torch.float32), to_dev(g, torch.bfloat16), to_dev(w, torch.float32)]
    dyd = to_dev(dy, torch.float32)
    r1 = gla.head_norm_gate_bwd(dyd, *args, 4)
    r2 = gla.head_norm_gate_bwd(dyd, *args, 4)
    assert all(torch.equal(a, b) for a, b in zip(r1, r2))


def test_head_norm_no_tokens(env):
    gla, torch = env
    e = torch.empty((0, 16, 192), device="cuda")
    w = torch.ones((4, 192), device="cuda")
    y, _ = gla.head_norm_gate(e, e, w, 4)
    _, _, dw = gla.head_norm_gate_bwd(e, e, e, w, 4)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.count_nonzero(dw).item() == 0
