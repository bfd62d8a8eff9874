"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import json
import os

import numpy as np
import pytest

from _pins import ALL_PINS, GOLDEN


@pytest.mark.parametrize("name", list(ALL_PINS))
def test_pin(olib, name):
    ok, detail = ALL_PINS[name](olib)
    assert ok, f"{name}: {detail}"


def test_printed_shapes_are_consistent():
    """The mixer sizes the page prints agree with one another and with the
    constants the synthetic workloads use."""
    import synth
    g = json.load(open(os.path.join(GOLDEN, "model_shapes_printed.json")))
    assert g["qkvg_width"] == g["H"] * (2 * g["d_k"] + 2 * g["d_v"])
    assert g["sequence"] == g["num_chunks"] * g["chunk"]
    assert (synth.DK, synth.DV, synth.CHUNK) == (g["d_k"], g["d_v"], g["chunk"])
    # per-sequence GLA state over all layers: 24 x 16 x 96 x 192 fp32 = 27 MiB
    assert g["layers"] * g["H"] * g["d_k"] * g["d_v"] * 4 == 27 * 2 ** 20


def test_oracle_threads_do_not_change_results(olib):
    import oracle
    r = np.random.default_rng(3)
    B, T, H, dk, dv = 3, 7, 4, 5, 6
    q, k, dO = r.standard_normal((B, T, H, dk)), r.standard_normal((B, T, H, dk)), None
    v = r.standard_normal((B, T, H, dv))
    dO = r.standard_normal((B, T, H, dv))
    a = r.standard_normal((H, dk))
    g = oracle.decay_schedule(H)
    o1, f1 = oracle.fwd(q, k, v, g, a, nthreads=1)
    o2, f2 = oracle.fwd(q, k, v, g, a, nthreads=5)
    b1 = oracle.bwd(q, k, v, g, a, dO, nthreads=1)
    b2 = oracle.bwd(q, k, v, g, a, dO, nthreads=7)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)
    assert all(np.array_equal(b1[n], b2[n]) for n in b1)


def test_oracle_rejects_bad_sizes(olib):
    import ctypes
    rc = olib.oracle_fwd(*([None] * 8), 1, 1, 0, 96, 192, 1)
    assert rc != 0
