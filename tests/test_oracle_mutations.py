"""The pins have teeth: a plausible mistake planted in a copy of the oracle's C source
(a wrong scale index or layout stride, a wrong exponent bias, a dropped or misplaced term, a
wrong sign, an off-by-one range, swapped nibbles) makes at least one pin of
test_oracle_pins.py fail.  Each mutant is built with the oracle's own compiler flags and
run through the pins in a child process (GMMFR_ORACLE_LIB points the oracle at it)."""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gmmfr_oracle.c")

# (name, text in gmmfr_oracle.c (exactly once), replacement)
MUTANTS = [
    ("token scale half from k/64", "k / 64) * 2 + (k / 32) % 2]);", "k / 64) * 2 + (k / 64) % 2]);"),
    ("transposed scale stride", "(n * Ks + k / 64) * 2", "(n + k / 64 * a->N) * 2"),
    ("E4M3 exponent bias", "e - 10); /* (1 + m/8)", "e - 11); /* (1 + m/8)"),
    ("E5M2 subnormal exponent", "ldexp((double)m, -16)", "ldexp((double)m, -15)"),
    ("E8M0 bias", "(int)code - 127", "(int)code - 126"),
    ("bf16 bit position", "(bits & 0xFFFFu) << 16", "(bits & 0xFFFFu) << 15"),
    ("E2M1 nibble order", "(i & 1) ? (b >> 4) : (b & 15)", "(i & 1) ? (b & 15) : (b >> 4)"),
    ("dropped logit", "out64[r * N + n0 + j] += lg * (acc[j] + b);", "out64[r * N + n0 + j] += acc[j] + b;"),
    ("bias after the logit", "out64[r * N + n0 + j] += lg * (acc[j] + b);",
     "out64[r * N + n0 + j] += lg * acc[j] + b;"),
    ("shared term subtracted", "out64[r * N + n] += a->shared_weight", "out64[r * N + n] -= a->shared_weight"),
    ("last K element dropped", "for (int64_t k = 0; k < K; ++k) {\n          const double av",
     "for (int64_t k = 0; k < K - 1; ++k) {\n          const double av"),
    ("count ranges restart at 0", "const int64_t s = prev_end;", "const int64_t s = 0;"),
    ("prefix-sum end off by one", "t = g < s ? s : (g > a->M ? a->M : g);",
     "t = g < s ? s : (g > a->M ? a->M : (g > s ? g - 1 : g));"),
]


def _build(tmp, i, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    d = os.path.join(tmp, f"m{i}")
    os.makedirs(d)
    open(os.path.join(d, "gmmfr_oracle.c"), "w").write(src.replace(old, new))
    shutil.copy(os.path.join(ROOT, "oracle", "gmmfr_oracle.h"), d)
    lib = os.path.join(d, "liboracle_mutant.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    os.path.join(d, "gmmfr_oracle.c"), "-o", lib, "-lm"], check=True)
    return lib


def _pins_fail(lib):
    env = dict(os.environ, GMMFR_ORACLE_LIB=lib, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    # a failed assertion, not a crash of the child
    return r.returncode == 1 and " failed" in r.stdout


def test_every_planted_mistake_fails_a_pin(tmp_path):
    import oracle
    oracle.build()
    # the unmodified source passes the pins through the same route
    libs = [_build(str(tmp_path), i, old, new) for i, (_, old, new) in enumerate(MUTANTS)]
    with cf.ThreadPoolExecutor(min(8, os.cpu_count() or 1)) as ex:
        caught = list(ex.map(_pins_fail, libs))
    survivors = [m[0] for m, c in zip(MUTANTS, caught) if not c]
    assert not survivors, f"mutants no pin catches: {survivors}"


def test_the_unmodified_source_passes_through_the_same_route(tmp_path):
    lib = _build(str(tmp_path), 0, "(int)code - 127", "(int)code - 127")
    env = dict(os.environ, GMMFR_ORACLE_LIB=lib, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-q",
                        "-p", "no:cacheprovider"], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
