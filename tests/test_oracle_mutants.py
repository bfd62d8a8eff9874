"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
each one fails at least one pin -- i.e. the pins can tell a wrong oracle."""
import os
import shutil

import pytest

import oracle
from _pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "gla_oracle.c")

# (name, text in the oracle, replacement, which occurrence (0-based))
MUTANTS = [
    ("fwd: no decay in the state update", "S[i * dv + n] = lam * S[i * dv + n] + k[i] * v[n];",
     "S[i * dv + n] = S[i * dv + n] + k[i] * v[n];", 0),
    ("fwd: aug term subtracted", "o[n] = acc + g * v[n];", "o[n] = acc - g * v[n];", 0),
    ("fwd: gate uses q*q", "z += a[i] * q[i] * k[i];", "z += a[i] * q[i] * q[i];", 0),
    ("gate is not the logistic function", "return 1.0 / (1.0 + exp(-z));",
     "return 1.0 / (1.0 + exp(z));", 0),
    ("fwd: init state of pair 0 for every pair", "memcpy(S, j->init + p * dk * dv,",
     "memcpy(S, j->init,", 0),
    ("bwd: dq misses the aug term", "dq[i] = acc + r * a[i] * k[i];", "dq[i] = acc;", 0),
    ("bwd: dk aug term uses k", "dk_out[i] = acc + r * a[i] * q[i];",
     "dk_out[i] = acc + r * a[i] * k[i];", 0),
    ("bwd: dv skip uses r", "dv_out[n] = acc + s * dO[n];", "dv_out[n] = acc + r * dO[n];", 0),
    ("bwd: d_init misses lambda", "j->dinit[p * dk * dv + i] = lam * G[i];",
     "j->dinit[p * dk * dv + i] = G[i];", 0),
    ("bwd: adjoint not decayed", "if (t < T - 1)\n                for (long i = 0; i < dk * dv; ++i) G[i] *= lam;",
     "", 0),
    ("bwd: d_a misses k", "da[i] += r * q[i] * k[i];", "da[i] += r * q[i];", 0),
    ("bwd: sigma' wrong", "double r = s * (1.0 - s) * dov;", "double r = s * dov;", 0),
    ("bwd: dq uses the state before the update",
     "S[i * dv + n] = lam * S[i * dv + n] + k[i] * v[n];\n            double z = 0.0, dov = 0.0;",
     "S[i * dv + n] = lam * S[i * dv + n];\n            double z = 0.0, dov = 0.0;", 0),
    ("decode: a of layer 0 for every layer", "const double *a = j->a + (l * j->H + h) * dk;",
     "const double *a = j->a + h * dk;", 0),
    ("decode: no decay", "S[i * dv + n] = lam * S[i * dv + n] + k[i] * v[n];",
     "S[i * dv + n] = S[i * dv + n] + k[i] * v[n];", 2),
    ("schedule: exponent h/H", "(double)h / (double)(H - 1)", "(double)h / (double)H", 0),
    ("schedule: base e instead of 2", "gamma[h] = -log(2.0) / half_life;",
     "gamma[h] = -1.0 / half_life;", 0),
]


def _replace_nth(s, old, new, n):
    idx = -1
    for _ in range(n + 1):
        idx = s.find(old, idx + 1)
        if idx < 0:
            raise AssertionError(f"mutation site not found: {old!r}")
    return s[:idx] + new + s[idx + len(old):]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, nth):
    src = open(SRC).read()
    mut = _replace_nth(src, old, new, nth)
    assert mut != src
    csrc = tmp_path / "mutant.c"
    csrc.write_text(mut)
    so = oracle.build(force=True, src=str(csrc), out=str(tmp_path / "libmutant.so"))
    lib = oracle.load(so)
    failed = []
    for pname, pin in ALL_PINS.items():
        try:
            ok, _ = pin(lib)
        except Exception:          # a crash on a wrong oracle also counts as caught
            ok = False
        if not ok:
            failed.append(pname)
    assert failed, f"mutant '{name}' passes every pin"
