"""bench.py end to end on a reduced workload (2 training sequences, a pool of 8 serving
sequences): it exits 0 and prints one JSON line with every key of the benchmark contract,
its rates derived from the batch it ran, its step counted in our own kernel launches and both
chunk calls also timed alone."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--batch", "2", "--n-seq", "8",
           "--steps", "3", "--warmup", "3", "--no-cpu-baseline"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["B"] == 2 and "B=2 " in d["config"]["workload"]
    assert d["config"]["decode_pool"][0] == 8
    # value = the tokens of the batch run over the chunk calls' time inside the step
    ms = d["parts_ms"]["chunk_fwd"] + d["parts_ms"]["chunk_bwd"]
    assert d["value"] == pytest.approx(2 * 2048 / (ms * 1e-3), rel=1e-6)
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in d["roofline"], key
    assert d["roofline"]["frac"] == pytest.approx(d["roofline"]["achieved"] / d["roofline"]["peak"])
    for name in ("roofline_chunk_fwd", "roofline_chunk_bwd"):
        alone = d[name]["alone"]
        assert alone["ms"] > 0 and alone["frac"] > 0
    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > 0
    assert e["h2d_bytes_per_step"] == 2 * 2048 * 16 * (96 + 96 + 192 + 192) * 2  # bf16 q,k,v,dO
    assert e["d2h_bytes_per_step"] == 16 * 96 * 4  # d_aug
    assert len(e["windows_s"]) == 3 and 0 < e["link"]["frac"]
    assert d["e2e_full_readback"]["d2h_bytes_per_step"] > e["d2h_bytes_per_step"]
    assert d["gpu_launches"] >= 4 * 3  # chunk fwd, chunk bwd, d_aug reduction, decode per step
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
