"""How sensitive the oracle's pins are: each case plants one plausible mistake
(a dropped term, a wrong sign, scale or index, a transposed operand, an eps
the pages' reading leaves out) in a copy of the float64 oracle's C source,
builds that copy on the CPU, and runs the pins of test_oracle.py against it
in a child process.  Every mutant must fail at least one pin.  The unchanged
copy, built and run the same way, must pass them all: that control shows the
harness itself works, so a caught mutant is caught by a pin and not by a
broken build.

The mutants touch the oracle only (test infrastructure); nothing here loads
the CUDA library."""
import os
import re
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "favor_oracle.c")

# name -> (text of the oracle source, the mistaken text put in its place);
# each original text occurs exactly once in the source.
MUTANTS = {
    "positive map: the -|x|^2/2 factor dropped":
        ("double pref = exp(-norm2 / 2.0) * scale;", "double pref = scale;"),
    "positive map: +|x|^2/2 instead of -|x|^2/2":
        ("double pref = exp(-norm2 / 2.0) * scale;", "double pref = exp(norm2 / 2.0) * scale;"),
    "feature scale 1/m instead of 1/sqrt(m)":
        ("double scale = 1.0 / sqrt((double)m);", "double scale = 1.0 / (double)m;"),
    "projection with omega transposed":
        ("proj += wi[j] * xt[j];", "proj += omega[(size_t)j * m + i] * xt[j];"),
    "trig map: cos in place of sin":
        ("pt[2 * i] = scale * sin(proj);", "pt[2 * i] = scale * cos(proj);"),
    "softmax-scaled trig: exp(|x|^2) instead of exp(|x|^2/2)":
        ("const double g = exp(norm2 / 2.0) * scale;", "const double g = exp(norm2) * scale;"),
    "elu+1: the +1 dropped":
        ("pt[j] = v > 0.0 ? v + 1.0 : exp(v);", "pt[j] = v > 0.0 ? v : exp(v);"),
    "causal: state built from the previous key (diagonal left out)":
        ("rc = oracle_features(k + (size_t)i * d, omega, 1, d, m, map, phik);",
         "rc = oracle_features(k + (size_t)(i > 0 ? i - 1 : 0) * d, omega, 1, d, m, map, phik);"),
    "causal: values read in reverse row order":
        ("const double *vi = v + (size_t)i * dv;", "const double *vi = v + (size_t)(L - 1 - i) * dv;"),
    "output: eps = 1e-6 added to the denominator":
        ("for (int c = 0; c < dv; ++c) oi[c] = oi[c] / den;",
         "for (int c = 0; c < dv; ++c) oi[c] = oi[c] / (den + 1e-6);"),
    "decode step: numerator not divided by the denominator":
        ("oh[c] = num / den;", "oh[c] = num;"),
    "carried state: sum of features not accumulated":
        ("zh[f] += phik[f];\n            }\n        }\n        free(phik);",
         "zh[f] += 0.0 * phik[f];\n            }\n        }\n        free(phik);"),
    "backward: wrong sign of the denominator gradient":
        ("dden[i] = -gdo / den;", "dden[i] = gdo / den;"),
    "backward, positive map: the -x sum term of dx dropped":
        ("for (int j = 0; j < d; ++j) dx[j] -= tot * x[j];", "for (int j = 0; j < d; ++j) dx[j] -= 0.0 * x[j];"),
    "Philox: the two products' high words swapped":
        ("uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;", "uint64_t n0 = hi0 ^ c1 ^ k0, n2 = hi1 ^ c3 ^ k1;"),
    "Gram-Schmidt: projection added instead of removed":
        ("for (int t = 0; t < d; ++t) v[t] -= dot * qj[t];", "for (int t = 0; t < d; ++t) v[t] += dot * qj[t];"),
    "block-orthogonal rows scaled by |g|^2 instead of |g|":
        ("const double chi = sqrt(ss);", "const double chi = ss;"),
    "forward: a flat head index decoded as [H][B] (the wrong head's omega)":
        ("int h = bh % H;", "int h = bh / B;"),
    "trig map: each pair stored as [cos, sin] (the output cannot see it)":
        ("pt[2 * i] = scale * sin(proj);\n                pt[2 * i + 1] = scale * cos(proj);",
         "pt[2 * i] = scale * cos(proj);\n                pt[2 * i + 1] = scale * sin(proj);"),
    "forward: a query's features taken from the key row":
        ("rc = oracle_features(q + (size_t)i * d, omega, 1, d, m, map, phiq);",
         "rc = oracle_features(k + (size_t)i * d, omega, 1, d, m, map, phiq);"),
}

# the child: point the oracle package at the copy's source and build folder,
# then run the pins
_DRIVER = r"""
import os, sys
root, src, bdir = sys.argv[1:4]
sys.path.insert(0, root)
import oracle
oracle._SRC = src
oracle._BUILD = bdir
oracle._LIB_PATH = os.path.join(bdir, "liboracle.so")
import pytest
sys.exit(pytest.main([os.path.join(root, "tests", "test_oracle.py"), "-x", "-q", "-m", "not gpu",
                      "-p", "no:cacheprovider", "-W", "ignore"]))
"""


def _mutated(name):
    text = open(SRC).read()
    if name is None:
        return text
    old, new = MUTANTS[name]
    assert text.count(old) == 1, f"mutation site of {name!r} not unique in the oracle source"
    return text.replace(old, new)


@pytest.fixture(scope="module")
def runs(tmp_path_factory):
    """Build and run every mutant (and the control) in child processes, as many
    at a time as the host has cores."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    jobs = []
    for i, name in enumerate([None] + list(MUTANTS)):
        d = tmp_path_factory.mktemp(f"mutant{i}")
        src = d / "favor_oracle.c"
        src.write_text(_mutated(name))
        jobs.append((name, [sys.executable, "-c", _DRIVER, ROOT, str(src), str(d / "_build")]))

    def run(job):
        name, cmd = job
        r = subprocess.run(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                           text=True, timeout=900)
        return name, (r.returncode, r.stdout)

    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as pool:
        return dict(pool.map(run, jobs))


def test_unchanged_copy_passes_every_pin(runs):
    rc, text = runs[None]
    assert rc == 0, text[-3000:]


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_the_mutant(runs, name):
    rc, text = runs[name]
    failed = re.findall(r"^FAILED (\S+)", text, re.M)
    # exit code 1: tests ran and one failed (not a crash, build or collection error)
    assert rc == 1 and failed, f"{name}: exit {rc}, no pin failed\n{text[-3000:]}"
