"""Plausible mistakes planted in copies of the oracle must each fail a pin.

Each mutant is the oracle's C source with one textual change (a dropped term,
a wrong sign, a wrong index or operand), compiled by gcc into a temporary
library and checked in a child process, so the real oracle is never touched."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = [
    ("dropped scale", "w[j] = J->scale * dot;", "w[j] = dot;"),
    ("causal mask off by one", "return i + 1 < Nk ? i + 1 : Nk;", "return i < Nk ? i : Nk;"),
    ("end-aligned mask without offset", "return i + 1 + (Nk - Nq);", "return i + 1;"),
    ("end-aligned offset reversed", "return i + 1 + (Nk - Nq);", "return i + 1 + (Nq - Nk);"),
    ("value used as key", "qi[c] * kh[j * J->d + c]", "qi[c] * vh[j * J->d + c]"),
    ("sign of exponent", "w[j] = exp(w[j] - m);", "w[j] = exp(m - w[j]);"),
    ("missing normalisation", "oi[c] /= l;", "oi[c] /= 1.0;"),
    ("lse without max", "m + log(l)", "log(l)"),
    ("max not subtracted", "w[j] = exp(w[j] - m);", "w[j] = exp(w[j]);"),
    ("subset row index", "(bh * J->Nq + i) * J->d", "(bh * J->Nq + r) * J->d"),
    ("values from head 0", "J->v + bh * J->Nk * J->d", "J->v + 0 * J->Nk * J->d"),
    ("one key dropped", "for (int64_t j = 0; j < nkeys; ++j)\n            for (int64_t c = 0; c < J->d; ++c) oi[c] +=",
     "for (int64_t j = 1; j < nkeys; ++j)\n            for (int64_t c = 0; c < J->d; ++c) oi[c] +="),
]


# Mistakes in the rotary embedding, each caught by the complex-number pin.
ROTARY_MUTANTS = [
    ("rotary sign of sin", "yr[ia] = a * c - b * s;", "yr[ia] = a * c + b * s;"),
    ("rotary cos and sin swapped", "yr[ib] = a * s + b * c;", "yr[ib] = a * c + b * s;"),
    ("rotary half-split partner", "interleaved ? 2 * i + 1 : i + half", "interleaved ? 2 * i + 1 : i + 1"),
    ("rotary table row ignored", "cos_t[n * half + i]", "cos_t[i]"),
]


# Mistakes in the backward pass, each caught by a backward pin.
BWD_MUTANTS = [
    ("softmax Jacobian without the row term", "const double ds = p[j] * (dp[j] - rowdot);",
     "const double ds = p[j] * dp[j];"),
    ("value gradient without the weights", "dvh[j * J->d + c] += p[j] * gi[c];", "dvh[j * J->d + c] += gi[c];"),
    ("key gradient unscaled", "dkh[j * J->d + c] += J->scale * ds * qi[c];", "dkh[j * J->d + c] += ds * qi[c];"),
    ("query gradient from values", "dqi[c] += J->scale * ds * kh[j * J->d + c];",
     "dqi[c] += J->scale * ds * vh[j * J->d + c];"),
    ("output gradient against keys", "dot += gi[c] * vh[j * J->d + c];", "dot += gi[c] * kh[j * J->d + c];"),
    ("row weights not normalised", "                p[j] /= l;\n", "\n"),
]


def _run_mutant(tmp_path, old, new, *mode):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not found once: {old!r}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-D_GNU_SOURCE",
                    str(path), "-o", str(lib), "-lm"], check=True)
    return subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_mutant_runner.py"), str(lib), *mode],
                          capture_output=True, text=True, timeout=300)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_fails_a_pin(tmp_path, name, old, new):
    res = _run_mutant(tmp_path, old, new)
    assert res.returncode == 1, f"mutant '{name}' survived every pin: {res.stdout}{res.stderr}"


@pytest.mark.parametrize("name,old,new", BWD_MUTANTS, ids=[m[0] for m in BWD_MUTANTS])
def test_bwd_mutant_fails_a_pin(tmp_path, name, old, new):
    res = _run_mutant(tmp_path, old, new, "bwd")
    assert res.returncode == 1, f"mutant '{name}' survived every backward pin: {res.stdout}{res.stderr}"


@pytest.mark.parametrize("name,old,new", ROTARY_MUTANTS, ids=[m[0] for m in ROTARY_MUTANTS])
def test_rotary_mutant_fails_the_pin(tmp_path, name, old, new):
    res = _run_mutant(tmp_path, old, new, "rotary")
    assert res.returncode == 1, f"mutant '{name}' survived: {res.stdout}{res.stderr}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    lib = tmp_path / "libcopy.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-D_GNU_SOURCE",
                    SRC, "-o", str(lib), "-lm"], check=True)
    for mode in ([], ["rotary"], ["bwd"]):
        res = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_mutant_runner.py"), str(lib), *mode],
                             capture_output=True, text=True, timeout=300)
        assert res.returncode == 0, res.stdout + res.stderr
