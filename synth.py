"""Seeded synthetic inputs for the Simple GLA mixer workloads.

Shared by the tests, the benchmark and the smoke check, so that the CUDA path
and the fp64 oracle see exactly the same numbers.  This module holds none of the
method's arithmetic: it only draws Gaussian tensors, applies the workload recipe
(q scaled by dk^-1/2, the stated standard deviations) and rounds to bf16.

Every tensor comes from its own PCG64 stream keyed by (seed, tensor id[, extra
keys]), so tensors do not depend on draw order or on one another's sizes.
"""
from __future__ import annotations

import numpy as np

DK, DV, CHUNK = 96, 192, 128

# tensor ids of the per-tensor streams
A, INIT, Q, K, V, DO, DFIN = 0, 1, 2, 3, 4, 5, 6
WARM_Q, WARM_K, WARM_V = 10, 11, 12


def normal(seed: int, tid: int, shape, std: float = 1.0, extra=()) -> np.ndarray:
    """float32 N(0, std^2) draws from the stream keyed (seed, tid, *extra)."""
    ss = np.random.SeedSequence([int(seed), int(tid), *[int(e) for e in extra]])
    g = np.random.Generator(np.random.PCG64(ss))
    x = g.standard_normal(size=tuple(shape), dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16, round-to-nearest-even; returns the raw uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values exactly representable in bf16 (what a bf16 input path sees)."""
    return bf16_to_f32(bf16_bits(x))


# --------------------------------------------------------------------------
# Workload recipes.  Shapes and distributions follow the pages' training shape
# (T=2048, H=16, dk=96, dv=192, chunk 128) and serving shape (1,280 concurrent
# sequences x 24 layers); the values are synthetic.

def qkv(seed: int, B: int, T: int, H: int, bf16: bool = True):
    """q ~ N(0,1)*dk^-1/2, k, v ~ N(0,1), token-major [B,T,H,d] (float32 values)."""
    q = normal(seed, Q, (B, T, H, DK)) * np.float32(DK ** -0.5)
    k = normal(seed, K, (B, T, H, DK))
    v = normal(seed, V, (B, T, H, DV))
    if bf16:
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    return q, k, v


def grad_out(seed: int, B: int, T: int, H: int, bf16: bool = True):
    d = normal(seed, DO, (B, T, H, DV))
    return round_bf16(d) if bf16 else d


def aug_balance(seed: int, shape, std: float):
    if std == 0.0:
        return np.zeros(shape, np.float32)
    return normal(seed, A, shape, std)


def init_state(seed: int, B: int, H: int, std: float):
    return normal(seed, INIT, (B, H, DK, DV), std)


def decode_warm_tokens(seed: int, seq: int, n_tokens: int, L: int, H: int):
    """The random tokens a decode state is warmed up with, for one sequence:
    q,k [n_tokens, L, H, dk], v [n_tokens, L, H, dv], float32."""
    q = normal(seed, WARM_Q, (n_tokens, L, H, DK), extra=(seq,)) * np.float32(DK ** -0.5)
    k = normal(seed, WARM_K, (n_tokens, L, H, DK), extra=(seq,))
    v = normal(seed, WARM_V, (n_tokens, L, H, DV), extra=(seq,))
    return q, k, v


def decode_token(seed: int, N: int, L: int, H: int, step: int = 0):
    """One new token per state: q,k [N,L,H,dk], v [N,L,H,dv], float32."""
    q = normal(seed, Q, (N, L, H, DK), extra=(step,)) * np.float32(DK ** -0.5)
    k = normal(seed, K, (N, L, H, DK), extra=(step,))
    v = normal(seed, V, (N, L, H, DV), extra=(step,))
    return q, k, v


# The five workloads.  "seed" keys every stream of that workload.
WORKLOADS = {
    "tiny_fp32": dict(B=1, T=256, H=2, dtype="fp32", a_std=0.1, init_std=0.0, seed=0,
                      bwd=True),
    "layer_fwd": dict(B=8, T=2048, H=16, dtype="bf16", a_std=0.0, init_std=0.0, seed=1,
                      bwd=False),
    "layer_fwd_aug": dict(B=8, T=2048, H=16, dtype="bf16", a_std=0.02, init_std=0.0, seed=101,
                          bwd=False),
    "train_fwd_bwd": dict(B=32, T=2048, H=16, dtype="bf16", a_std=0.02, init_std=0.0, seed=2,
                          bwd=True),
    "long_prefill": dict(B=2, T=131072, H=16, dtype="bf16", a_std=0.02, init_std=0.01, seed=4,
                         bwd=False),
}
DECODE = dict(N=1280, L=24, H=16, warm_tokens=64, a_std=0.02, seed=3, steps=100)


def chunk_inputs(name: str, B: int | None = None, T: int | None = None):
    """All inputs of a chunked workload (optionally with B or T overridden for a
    smaller case of the same recipe).  float32 arrays; bf16 workloads hold
    bf16-representable values."""
    c = dict(WORKLOADS[name])
    if B is not None:
        c["B"] = B
    if T is not None:
        c["T"] = T
    bf16 = c["dtype"] == "bf16"
    s, Bn, Tn, H = c["seed"], c["B"], c["T"], c["H"]
    out = dict(cfg=c)
    out["a"] = aug_balance(s, (H, DK), c["a_std"])
    out["init_state"] = init_state(s, Bn, H, c["init_std"]) if c["init_std"] > 0 else None
    out["q"], out["k"], out["v"] = qkv(s, Bn, Tn, H, bf16)
    if c["bwd"]:
        out["dO"] = grad_out(s, Bn, Tn, H, bf16)
    return out
