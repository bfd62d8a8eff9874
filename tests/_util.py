"""Helpers shared by the tests: the parity metric and host<->device marshalling."""
from __future__ import annotations

import numpy as np

# Parity bars: max|x - ref| / rms(ref) per output tensor.
TOL_CHUNK = 2e-2   # bf16 / fp16 / fp32 inputs through the tensor-core path
TOL_DECODE = 1e-4  # fp32 decode step


def rel_err(x, ref) -> float:
    """max|x - ref| / rms(ref); the absolute max error if ref is identically zero."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if not np.all(np.isfinite(x)):
        return float("inf")
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = float(np.abs(x - ref).max()) if x.size else 0.0
    return err / rms if rms > 0 else err


def to_dev(x, dtype, device="cuda"):
    """float32 numpy -> torch tensor of `dtype` on the device (bf16 values must already be
    bf16-representable so the conversion is exact)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device).to(dtype)


def as_dtype_values(x, name: str):
    """The float32 values a kernel sees for an input of type `name` (bf16 / fp16 / fp32)."""
    import synth
    if name == "bf16":
        return synth.round_bf16(x)
    if name == "fp16":
        return x.astype(np.float16).astype(np.float32)
    return np.asarray(x, np.float32)


def oracle_decays(H: int, t_min: float = 1.0, t_max: float = 2048.0):
    """The oracle's log-decays rounded to fp32, for both sides of a parity test: returns
    (a host float32 torch tensor [H] for the library, the same values as fp64 numpy for the
    oracle).  The library's own schedule is checked against these values separately."""
    import torch

    import oracle
    g32 = oracle.decay_schedule(H, t_min, t_max).astype(np.float32)
    return torch.from_numpy(g32.copy()), g32.astype(np.float64)
