"""The allocation-free backward, gla_chunk_bwd_noalloc, called through the C ABI.

It is meant for callers that cannot give the library a device buffer (allocation forbidden
inside their execution callback, memory reserved in full up front, or no cudaMalloc/cudaFree
allowed in a latency-critical loop): it keeps its scratch in a fixed array inside the
library.  Its results must equal those of gla_chunk_bwd, which takes a caller workspace,
and stay equal when the shared array is reused by the next call.  This file is collected
last so that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import synth
from _util import TOL_CHUNK, rel_err, to_dev, oracle_decays

GLA_ERR_UNSUPPORTED, GLA_ERR_WORKSPACE = 2, 7
MAX_BH = 2048
A16 = 0x1000  # a 16-byte aligned stand-in pointer, never dereferenced by the size checks


def _lib():
    import gated_linear_attention_chunked_gb300 as gla
    from gated_linear_attention_chunked_gb300 import _build
    _build.build()
    lib = gla.load()
    fn = lib.gla_chunk_bwd_noalloc
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] + [ctypes.c_void_p] * 11 + \
        [ctypes.c_int] * 5 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return gla, fn


def test_noalloc_rejects_sizes_beyond_its_array_and_fp32_inputs():
    _, fn = _lib()
    args = [A16] * 3 + [0] + [A16] * 11
    # B * H = 2049 > the fixed scratch: refused before anything is launched
    assert fn(*args, 2049, 128, 1, 96, 192, None) == GLA_ERR_WORKSPACE
    assert fn(*args, 129, 128, 16, 96, 192, None) == GLA_ERR_WORKSPACE
    # fp32 inputs would need a workspace for their fp16 copies
    args[3] = 1
    assert fn(*args, 1, 128, 1, 96, 192, None) == GLA_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_on_two_calls_in_a_row():
    import torch

    import oracle
    assert torch.cuda.is_available(), "GPU test without a CUDA device"
    gla, fn = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    # problems back to back, each reusing the array the one before wrote: bf16 and fp16
    # inputs, a ragged last chunk, and B * H exactly at the array's limit (its last rows
    # written and read)
    cases = [(2, 384, 5, 41, "bf16"), (3, 256, 16, 42, "fp16"), (2, 200, 3, 43, "bf16"),
             (MAX_BH // 16, 128, 16, 44, "bf16"), (1, 300, 2, 45, "fp16")]
    for (B, T, H, seed, dt) in cases:
        td = torch.bfloat16 if dt == "bf16" else torch.float16
        code = gla.GLA_BF16 if dt == "bf16" else gla.GLA_FP16
        q, k, v = synth.qkv(seed, B, T, H, bf16=dt == "bf16")
        dO = synth.grad_out(seed, B, T, H, bf16=dt == "bf16")
        if dt == "fp16":  # the values an fp16 input holds
            q, k, v, dO = (x.astype(np.float16).astype(np.float32) for x in (q, k, v, dO))
        a = synth.aug_balance(seed, (H, 96), 0.1)
        init = synth.init_state(seed, B, H, 0.05)
        dfin = synth.normal(seed, synth.DFIN, (B, H, 96, 192), 0.05)
        qd, kd, vd, gd = (to_dev(x, td) for x in (q, k, v, dO))
        ad, id_, fd = (to_dev(x, torch.float32) for x in (a, init, dfin))
        gam, gam64 = oracle_decays(H)
        gam = gam.cuda()
        ref = gla.chunk_bwd(qd, kd, vd, gam, ad, gd, id_, fd)  # with a caller workspace
        f32 = dict(dtype=torch.float32, device="cuda")
        out = [torch.full((B, T, H, 96), float("nan"), **f32),
               torch.full((B, T, H, 96), float("nan"), **f32),
               torch.full((B, T, H, 192), float("nan"), **f32),
               torch.full((H, 96), float("nan"), **f32),
               torch.full((B, H, 96, 192), float("nan"), **f32)]
        rc = fn(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), code, gam.data_ptr(),
                ad.data_ptr(), id_.data_ptr(), gd.data_ptr(), fd.data_ptr(), None,
                *[x.data_ptr() for x in out], B, T, H, 96, 192, stream)
        assert rc == 0, gla.status_string(rc)
        torch.cuda.synchronize()
        assert gla.get_device_error() == 0
        names = ("dq", "dk", "dv", "d_aug", "d_init_state")
        for name, x, r in zip(names, out, ref):
            e = rel_err(x.cpu().numpy(), r.cpu().numpy())
            assert e <= TOL_CHUNK, f"{name}: {e:.3e}"
        # and against the fp64 oracle: every sequence of the small cases; at the array's
        # limit, its last two sequences (whose d_aug rows end the array) and the summed d_aug
        bs = slice(B - 2, B) if B * H == MAX_BH else slice(0, B)
        g = oracle.bwd(q[bs], k[bs], v[bs], gam64, a, dO[bs], init[bs], dfin[bs])
        errs = {}
        for name, key, x in zip(names, ("dq", "dk", "dv", "d_a", "d_init_state"), out):
            xs = x.cpu().numpy() if name == "d_aug" else x[bs].cpu().numpy()
            if name == "d_aug" and B * H == MAX_BH:
                continue  # summed over all B: compared with the workspace call above
            errs[name] = rel_err(xs, g[key])
            assert errs[name] <= TOL_CHUNK, f"{name} vs oracle: {errs[name]:.3e}"
        same = all(torch.equal(x, r) for x, r in zip(out, ref))
        print(f"no-alloc bwd B={B} T={T} H={H} {dt}: "
              f"{'bit-identical to' if same else 'within tolerance of'} the workspace call; "
              "oracle " + " ".join(f"{n} {e:.1e}" for n, e in errs.items()))
