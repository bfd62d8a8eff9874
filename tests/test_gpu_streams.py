"""Two independent problems on two CUDA streams at once give the same bits as the same calls
made one after the other: the chunked forward and backward (pairs cut into parts, the passes
beside the whole pairs, saved activations), the slice sums and the decode step keep no state
between calls or streams beyond the caller's buffers.  (The scratch-free backward shares one
library array by design and is not part of this.)"""
import numpy as np
import pytest

import synth
from _util import to_dev, oracle_decays

pytestmark = pytest.mark.gpu


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


def _problem(torch, seed, B, T, H):
    q, k, v = synth.qkv(seed, B, T, H)
    dO = synth.grad_out(seed, B, T, H)
    a = synth.aug_balance(seed, (H, 96), 0.1)
    init = synth.init_state(seed, B, H, 0.05)
    st = synth.normal(seed, synth.INIT, (B, H, 96, 192), 0.05)
    return dict(q=to_dev(q, torch.bfloat16), k=to_dev(k, torch.bfloat16),
                v=to_dev(v, torch.bfloat16), dO=to_dev(dO, torch.bfloat16),
                a=to_dev(a, torch.float32), init=to_dev(init, torch.float32),
                st=to_dev(st, torch.float32), gam=oracle_decays(H)[0].cuda(), B=B, T=T, H=H)


def _work(gla, torch, p, stream):
    """fwd (saving gate and copies) + bwd reading them + a slice sum + decode steps, all on
    `stream`; returns the outputs."""
    B, T, H = p["B"], p["T"], p["H"]
    with torch.cuda.stream(stream):
        gate = torch.empty(B, H, T, device="cuda")
        saved = torch.empty(gla.chunk_saved_states_size(B, T, H), dtype=torch.uint8,
                            device="cuda")
        o, fin = gla.chunk_fwd(p["q"], p["k"], p["v"], p["gam"], p["a"], p["init"], gate=gate,
                               saved_states=saved, stream=stream)
        g = gla.chunk_bwd(p["q"], p["k"], p["v"], p["gam"], p["a"], p["dO"], p["init"],
                          gate=gate, saved_states=saved, stream=stream)
        U = gla.chunk_state_sum(p["k"], p["v"], p["gam"], stream=stream)
        st = p["st"].view(B, 1, H, 96, 192).clone()  # one layer of B sequences' states
        a1 = p["a"].view(1, H, 96)
        outs = []
        for t in range(3):
            tok = [p[n][:, t].float().reshape(B, 1, H, -1).contiguous() for n in ("q", "k", "v")]
            od = torch.empty(B, 1, H, 192, device="cuda")
            gla.decode_step(st, *tok, p["gam"], a1, out=od, stream=stream)
            outs.append(od)
    return [o, fin, gate, *g, U, st, *outs]


def test_two_streams_match_one_after_the_other(env):
    gla, torch = env
    gla.set_split_parts(3)
    try:
        p1 = _problem(torch, 991, 10, 512, 16)  # 160 pairs: the passes beside a wave of them
        p2 = _problem(torch, 992, 3, 700, 8)
        s0 = torch.cuda.current_stream()
        seq = [_work(gla, torch, p, s0) for p in (p1, p2)]
        torch.cuda.synchronize()
        seq = [[x.cpu() for x in r] for r in seq]
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        for _ in range(3):  # several rounds, the two streams' calls interleaved
            par = [_work(gla, torch, p1, sa), _work(gla, torch, p2, sb)]
            torch.cuda.synchronize()
            assert gla.get_device_error() == 0
            for r_seq, r_par in zip(seq, par):
                for x, y in zip(r_seq, r_par):
                    assert torch.equal(x, y.cpu())
    finally:
        gla.set_split_parts(0)
