"""The pins catch plausible mistakes in the oracle.

Each case copies the oracle's C source, plants one mistake (a dropped term,
a wrong sign, a transposed operand, a wrong index, a wrong normaliser),
builds the copy and runs the quick pins against it: at least one pin must
fail.  The unmodified oracle passes all of them (test_oracle_pins.py).
This follows the "debugging tool must debug itself" advice of the
ops-debug page (sec. 7.2): checkers are validated on deliberately wrong
operators.
"""
import os
import shutil

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "gmm_oracle.c")

MUTANTS = [
    ("drop log-det term", "- 0.5 * c->logdet[k] ", ""),
    ("wrong sign of d2", "c->logpi[k] - 0.5 * d2", "c->logpi[k] + 0.5 * d2"),
    ("drop D/2 log 2pi", "- 0.5 * D * LOG_2PI", ""),
    ("transposed Cholesky factor in the solve", "v -= L[i * D + j] * work[j]",
     "v -= L[j * D + i] * work[j]"),
    ("solve divides by the wrong pivot", "work[i] = v / L[i * D + i]", "work[i] = v / L[0]"),
    ("Cholesky multiplies by the pivot", "L[i * D + j] = v / ljj;", "L[i * D + j] = v * ljj;"),
    ("log-det not doubled", "c->logdet[k] = 2.0 * ld;", "c->logdet[k] = ld;"),
    ("diag divides by sd not var", "d2 += t * t / v[d];", "d2 += t * t / sqrt(v[d]);"),
    ("iso log-det not scaled by D", "cov == O_DIAG ? ld : D * ld", "ld"),
    ("lse drops the max", "return m + log(s);", "return log(s);"),
    ("pi' normalised by K", "pi_out[k] = s0[k] / (double)N;", "pi_out[k] = s0[k] / (double)K;"),
    ("mean not normalised", "s1[(size_t)k * D + d] / s0[k]", "s1[(size_t)k * D + d] / (double)N"),
    ("second moment about the old mean", "y[d] = x[d] - mun[(size_t)k * D + d];",
     "y[d] = x[d] - mu[(size_t)k * D + d];"),
    ("iso variance not divided by D", "double v = acc / ((double)D * s0[k]);",
     "double v = acc / s0[k];"),
    ("gamma without normaliser", "double g = exp(l[k] - lse);\n        my0[k] += g;",
     "double g = exp(l[k]);\n        my0[k] += g;"),
    ("top-m ties to the higher index", "if (best < 0 || l[k] > l[best]) best = k;",
     "if (best < 0 || l[k] >= l[best]) best = k;"),
    ("weight dropped from the log joint", "c->logpi[k] = pi[k] > 0.0 ? log(pi[k]) : -INFINITY;",
     "c->logpi[k] = 0.0;"),
    ("ridge constant wrong", "add + 1e-3 * tr / D", "add + 1e-2 * tr / D"),
    ("full covariance stats use x not x-mu", "o[(size_t)a * D + b] += g * y[a] * y[b];",
     "o[(size_t)a * D + b] += g * x[a] * x[b];"),
    ("stored fp16 exponent off by one", "ldexp((double)(m | 0x400), e - 25)",
     "ldexp((double)(m | 0x400), e - 24)"),
    ("stored fp16 subnormal scale", "ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    ("stored bf16 mantissa width", "ldexp((double)(m | 0x80), e - 134)",
     "ldexp((double)(m | 0x100), e - 134)"),
]


def _run_pins(L):
    failed = []
    for name, fn in P.ALL_QUICK_PINS:
        try:
            fn(L)
        except AssertionError:
            failed.append(name)
    return failed


@pytest.mark.parametrize("desc,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, desc, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not unique: %r" % old
    mutated = tmp_path / "gmm_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(str(mutated), str(tmp_path / "libmutant.so")))
    failed = _run_pins(lib)
    assert failed, "no pin caught the mutant: " + desc


def test_unmutated_passes_all():
    assert _run_pins(oracle.lib()) == []
