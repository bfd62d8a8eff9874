"""The calls can be captured into a CUDA graph: a chunked forward and backward of a ragged
shape whose pairs are cut into parts (so the segment passes are in the graph too) and a decode
step, captured once and replayed on new inputs copied into the captured buffers, give exactly
the results of the same calls made eagerly on those inputs."""
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
    return gla, torch


def _inputs(seed, B, T, H):
    q, k, v = synth.qkv(seed, B, T, H)
    dO = synth.grad_out(seed, B, T, H)
    init = synth.init_state(seed, B, H, 0.05)
    dfin = synth.normal(seed, synth.DFIN, (B, H, 96, 192), 0.05)
    return q, k, v, dO, init, dfin


def test_capture_and_replay_matches_eager(env):
    gla, torch = env
    B, T, H, N, L = 2, 600, 3, 5, 2
    gla.set_split_parts(3)  # cut every pair into 3 parts: the segment passes run in the graph
    try:
        a = to_dev(synth.aug_balance(1, (H, 96), 0.1), torch.float32)
        gam = oracle_decays(H)[0].cuda()
        bufs = [to_dev(x, torch.bfloat16) for x in _inputs(1, B, T, H)[:4]]
        inits = [to_dev(x, torch.float32) for x in _inputs(1, B, T, H)[4:]]
        rng = np.random.default_rng(2)
        state = to_dev(rng.standard_normal((N, L, H, 96, 192)) * 0.3, torch.float32)
        tok = [to_dev(rng.standard_normal((N, L, H, d)), torch.float32) for d in (96, 96, 192)]
        ad = to_dev(synth.aug_balance(2, (L, H, 96), 0.02), torch.float32)

        def step(state_buf):
            q, k, v, dO = bufs
            o, fin = gla.chunk_fwd(q, k, v, gam, a, inits[0])
            g = gla.chunk_bwd(q, k, v, gam, a, dO, inits[0], inits[1])
            od = gla.decode_step(state_buf, tok[0], tok[1], tok[2], gam, ad)
            return [o, fin, *g, od]

        # eager first: every module is loaded before the capture
        step(state.clone())
        torch.cuda.synchronize()
        graph_state = state.clone()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step(graph_state.clone())  # warm-up on the capture stream
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            outs = step(graph_state)
        for seed in (3, 4):  # new inputs into the captured buffers, then replay
            new = _inputs(seed, B, T, H)
            for dst, x in zip(bufs, new[:4]):
                dst.copy_(to_dev(x, torch.bfloat16))
            for dst, x in zip(inits, new[4:]):
                dst.copy_(to_dev(x, torch.float32))
            for t_ in tok:
                t_.copy_(to_dev(rng.standard_normal(tuple(t_.shape)), torch.float32))
            before = graph_state.clone()
            graph.replay()
            ref = step(before)  # the same calls, eager, on the same inputs and state
            torch.cuda.synchronize()
            assert gla.get_device_error() == 0
            names = ("o", "final", "dq", "dk", "dv", "d_aug", "d_init", "decode_o")
            for name, x, r in zip(names, outs, ref):
                assert torch.equal(x, r), f"{name} differs between replay and eager"
            assert torch.equal(graph_state, before), "decode state differs between replay and eager"
        print(f"graph replay B={B} T={T} H={H} (3 parts) + decode {N}x{L}x{H}: bit-identical to eager")
    finally:
        gla.set_split_parts(0)
