"""Planted mistakes: the oracle's pins must catch each one.

Each case copies the ``oracle`` package into a temporary directory, plants one
plausible slip in the copy of ``bdla_oracle.c`` (a wrong sign, a dropped term,
a wrong operand, the decay applied after instead of before the update, a wrong
gate derivative, an adjoint that is not decayed, a checkpoint window read from
the wrong place, an ignored initial state), and runs the pins of the function
it lives in (``test_oracle_pins.py`` for the scalar decay,
``test_oracle_vec_pins.py`` for the per-channel decay,
``test_oracle_delta_pins.py`` for the gated delta rule) against the copy in a
fresh interpreter.  The pins pass on an unmodified copy and fail on every
mutant.  The committed oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")
VEC_PINS = os.path.join(ROOT, "tests", "test_oracle_vec_pins.py")
DELTA_PINS = os.path.join(ROOT, "tests", "test_oracle_delta_pins.py")

# (name, text in bdla_oracle.c, replacement[, occurrence]): the text occurs
# exactly once, or, where the scalar and per-channel functions share a line,
# the given occurrence (1 = first in the file) is replaced
MUTANTS = [
    ("sigmoid of -a", "return b / (1.0 + exp(-a));", "return b / (1.0 + exp(a));"),
    ("softplus term subtracted", "return -(fmax(a, 0.0) + log1p(exp(-fabs(a))));",
     "return -(fmax(a, 0.0) - log1p(exp(-fabs(a))));"),
    ("gate derivative without (1 - s)", "return b * s * (1.0 - s);", "return b * s;"),
    ("decay applied after the update", "Si[j] = g * Si[j] + ki * vt[j];",
     "Si[j] = g * (Si[j] + ki * vt[j]);"),
    ("output reads k instead of q", "const double qi = qt[i];", "const double qi = kt[i];", 1),
    ("initial state ignored in the forward",
     "memcpy(S, h0 + (size_t)u * ssz, ssz * sizeof(double));\n"
     "            else\n"
     "                memset(S, 0, ssz * sizeof(double));\n"
     "            for (int64_t t = cu[n];",
     "memset(S, 0, ssz * sizeof(double));\n"
     "            else\n"
     "                memset(S, 0, ssz * sizeof(double));\n"
     "            for (int64_t t = cu[n];", 1),
    ("dq drops the current token", "acc += (g * Sp[(size_t)i * dv + j] + kt[i] * vt[j]) * gt[j];",
     "acc += g * Sp[(size_t)i * dv + j] * gt[j];"),
    ("dq with an undecayed previous state", "acc += (g * Sp[(size_t)i * dv + j] + kt[i] * vt[j]) * gt[j];",
     "acc += (Sp[(size_t)i * dv + j] + kt[i] * vt[j]) * gt[j];"),
    ("dk reads dO instead of v", "acc += D[(size_t)i * dv + j] * vt[j];",
     "acc += D[(size_t)i * dv + j] * gt[j];", 1),
    ("dv reads q instead of k", "dvt[j] += D[(size_t)i * dv + j] * kt[i];",
     "dvt[j] += D[(size_t)i * dv + j] * qt[i];", 1),
    ("da without the gate factor g", "da[tt * H + h] = g * dot * log_decay_deriv(at, b, mode);",
     "da[tt * H + h] = dot * log_decay_deriv(at, b, mode);"),
    ("adjoint not decayed", "D[e] *= g;", "D[e] *= 1.0;"),
    ("every window restarts from the first checkpoint",
     "memcpy(S, ck + (size_t)w * ssz, ssz * sizeof(double));", "memcpy(S, ck, ssz * sizeof(double));", 1),
]

# the per-channel decay (fwd_vec / bwd_vec), checked by its own pins
GI = "const double gi = exp(log_decay(at[i], b, mode));"
VEC_MUTANTS = [
    ("state row decays by the next channel's gate", GI,
     "const double gi = exp(log_decay(at[(i + 1) % dk], b, mode));", 1),
    ("every row decays by channel 0's gate", GI, "const double gi = exp(log_decay(at[0], b, mode));", 1),
    ("backward window recomputed with channel 0's gate", GI,
     "const double gi = exp(log_decay(at[0], b, mode));", 3),
    ("vector dq with channel 0's gate", "acc += (g[i] * Sp[(size_t)i * dv + j] + kt[i] * vt[j]) * gt[j];",
     "acc += (g[0] * Sp[(size_t)i * dv + j] + kt[i] * vt[j]) * gt[j];"),
    ("vector dk reads dO instead of v", "acc += D[(size_t)i * dv + j] * vt[j];",
     "acc += D[(size_t)i * dv + j] * gt[j];", 2),
    ("vector da without the gate factor", "dat[i] = g[i] * dot * log_decay_deriv(at[i], b, mode);",
     "dat[i] = dot * log_decay_deriv(at[i], b, mode);"),
    ("vector adjoint not decayed", "D[(size_t)i * dv + j] *= g[i];", "D[(size_t)i * dv + j] *= 1.0;"),
    ("vector output reads k instead of q", "const double qi = qt[i];", "const double qi = kt[i];", 2),
]


# the gated delta rule (fwd_delta / bwd_delta), checked by its own pins
DELTA_MUTANTS = [
    ("delta retrieval not decayed", "e[j] = vt[j] - g * r;", "e[j] = vt[j] - r;", 1),
    ("delta projection built from q", "r += S[(size_t)i * dv + j] * kt[i];", "r += S[(size_t)i * dv + j] * qt[i];", 1),
    ("delta write strength applied twice", "S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + bt * kt[i] * e[j];",
     "S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + bt * bt * kt[i] * e[j];", 1),
    ("delta backward: retrieval adjoint without the gate", "dr[j] = -g * de[j];", "dr[j] = -de[j];"),
    ("delta backward: state adjoint misses the projection", "D[(size_t)i * dv + j] = g * D[(size_t)i * dv + j] + kt[i] * dr[j];",
     "D[(size_t)i * dv + j] = g * D[(size_t)i * dv + j];"),
    ("delta backward: dbeta from v instead of e", "De += D[(size_t)i * dv + j] * e[j];",
     "De += D[(size_t)i * dv + j] * vt[j];"),
    ("delta backward: decay gradient misses the retrieval term", "g * (dot - rde) * log_decay_deriv",
     "g * dot * log_decay_deriv"),
    ("delta backward: dk misses S dr", "dkt[i] = bt * De + Sdr;", "dkt[i] = bt * De;"),
]


def _copy_oracle(dst, mutation=None):
    pkg = os.path.join(dst, "oracle")
    os.makedirs(pkg)
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), pkg)
    with open(os.path.join(ROOT, "oracle", "bdla_oracle.c")) as f:
        src = f.read()
    if mutation is not None:
        old, new, nth = mutation
        if nth == 0:
            assert src.count(old) == 1, f"mutation site not unique or gone: {old!r}"
            src = src.replace(old, new)
        else:
            at = -1
            for _ in range(nth):
                at = src.find(old, at + 1)
                assert at >= 0, f"mutation site {old!r} has fewer than {nth} occurrences"
            src = src[:at] + new + src[at + len(old):]
    with open(os.path.join(pkg, "bdla_oracle.c"), "w") as f:
        f.write(src)


def _run_pins(cwd, pins=PINS):
    """The pins in a fresh interpreter whose `import oracle` finds the copy in
    cwd (no conftest, so the repository root is not put ahead of it)."""
    env = dict(os.environ, OMP_NUM_THREADS="2")
    env.pop("PYTHONPATH", None)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "--noconftest", "-p", "no:cacheprovider",
                           pins], cwd=cwd, env=env, capture_output=True, text=True, timeout=600)


def test_unmodified_copy_passes_the_pins(tmp_path):
    _copy_oracle(str(tmp_path))
    where = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"], cwd=str(tmp_path),
                           capture_output=True, text=True, timeout=120)
    assert where.stdout.strip().startswith(str(tmp_path)), where.stdout + where.stderr
    for pins in (PINS, VEC_PINS, DELTA_PINS):
        r = _run_pins(str(tmp_path), pins)
        assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


CASES = ([(m, PINS) for m in MUTANTS] + [(m, VEC_PINS) for m in VEC_MUTANTS] +
         [(m, DELTA_PINS) for m in DELTA_MUTANTS])


@pytest.mark.parametrize("mutant,pins", CASES, ids=[c[0][0] for c in CASES])
def test_pins_catch_planted_mistake(tmp_path, mutant, pins):
    name, old, new = mutant[:3]
    nth = mutant[3] if len(mutant) > 3 else 0
    _copy_oracle(str(tmp_path), (old, new, nth))
    r = _run_pins(str(tmp_path), pins)
    # 1 = some pin failed (not a crash, not a collection error)
    assert r.returncode == 1, f"{name}: pins returned {r.returncode}\n" + r.stdout[-3000:] + r.stderr[-2000:]
    assert " failed" in r.stdout, r.stdout[-3000:]
