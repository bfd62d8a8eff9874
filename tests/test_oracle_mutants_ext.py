"""Plant plausible mistakes in copies of the numpy oracles (state-pool decode, output epilogue,
causal conv) and check that each one fails at least one of their pins -- the pins can tell a
wrong oracle.  A mutant is a copy of oracle/__init__.py with one edit, loaded as a separate
module and handed to the pin tests in place of the oracle."""
import inspect
import types

import pytest

import oracle
import test_oracle_conv
import test_oracle_head_norm
import test_oracle_paged

# (name, text in oracle/__init__.py, replacement, which occurrence (0-based), pin module)
MUTANTS = [
    ("norm: sum instead of mean", "r = 1.0 / np.sqrt(np.mean(o * o, axis=-1) + eps)",
     "r = 1.0 / np.sqrt(np.sum(o * o, axis=-1) + eps)", 0, test_oracle_head_norm),
    ("norm: eps outside the root", "r = 1.0 / np.sqrt(np.mean(o * o, axis=-1) + eps)",
     "r = 1.0 / (np.sqrt(np.mean(o * o, axis=-1)) + eps)", 0, test_oracle_head_norm),
    ("norm: tiers interleaved", "return np.arange(H) // (H // n_tiers)",
     "return np.arange(H) % n_tiers", 0, test_oracle_head_norm),
    ("gate: sigmoid instead of SiLU", "silu = g / (1.0 + np.exp(-g))",
     "silu = 1.0 / (1.0 + np.exp(-g))", 0, test_oracle_head_norm),
    ("norm bwd: no projection term",
     "d_o = r * (dn - n * np.mean(dn * n, axis=-1, keepdims=True))", "d_o = r * dn", 0,
     test_oracle_head_norm),
    ("norm bwd: dg misses SiLU's slope", "dg = dy * n * wt * sg * (1.0 + g * (1.0 - sg))",
     "dg = dy * n * wt * sg", 0, test_oracle_head_norm),
    ("norm bwd: weight gradient to the wrong tier", "d_w[tier[h]] += per_head[h]",
     "d_w[h % n_tiers] += per_head[h]", 0, test_oracle_head_norm),
    ("conv: taps reversed", "z += w[:, j] * xe[:, j:j + T]", "z += w[:, 3 - j] * xe[:, j:j + T]",
     0, test_oracle_conv),
    ("conv: state one token early", "xe[:, T:T + 3].copy()", "xe[:, T - 1:T + 2].copy()", 0,
     test_oracle_conv),
    ("conv: bias dropped", "z = np.zeros((B, T, D)) if bias is None else",
     "z = np.zeros((B, T, D)) if True else", 0, test_oracle_conv),
    ("conv bwd: dx taps reversed", "dxe[:, j:j + T] += w[:, j] * dz",
     "dxe[:, j:j + T] += w[:, 3 - j] * dz", 0, test_oracle_conv),
    ("conv bwd: SiLU slope wrong", "dz = dy * sg * (1.0 + z * (1.0 - sg))", "dz = dy * sg", 0,
     test_oracle_conv),
    ("paged: layer offset ignored", "new[page, layer0:layer0 + L] = st", "new[page, 0:L] = st", 0,
     test_oracle_paged),
    ("paged: results to the pages in sorted order", "new[page, layer0:layer0 + L] = st",
     "new[np.sort(page), layer0:layer0 + L] = st", 0, test_oracle_paged),
]


def _replace_nth(s, old, new, n):
    idx = -1
    for _ in range(n + 1):
        idx = s.find(old, idx + 1)
        if idx < 0:
            raise AssertionError(f"mutation site not found: {old!r}")
    return s[:idx] + new + s[idx + len(old):]


def _run_pins(mod, pins):
    """Run every test function of the pin module against `mod`; return the names that failed."""
    failed = []
    saved = pins.oracle
    pins.oracle = mod
    try:
        for name, fn in inspect.getmembers(pins, inspect.isfunction):
            if not name.startswith("test_"):
                continue
            params = inspect.signature(fn).parameters
            calls = [dict(n_tiers=t) for t in (1, 2, 4)] if "n_tiers" in params else [dict()]
            for kw in calls:
                try:
                    fn(**kw)
                except AssertionError:
                    failed.append(name)
                    break
    finally:
        pins.oracle = saved
    return failed


def test_pins_pass_on_the_oracle():
    for pins in (test_oracle_conv, test_oracle_head_norm, test_oracle_paged):
        assert _run_pins(oracle, pins) == []


@pytest.mark.parametrize("name,old,new,nth,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, nth, pins):
    src = open(oracle.__file__).read()
    mut = _replace_nth(src, old, new, nth)
    assert mut != src
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = oracle.__file__
    exec(compile(mut, oracle.__file__, "exec"), mod.__dict__)
    failed = _run_pins(mod, pins)
    assert failed, f"no pin caught: {name}"
    print(f"{name}: caught by {failed}")
