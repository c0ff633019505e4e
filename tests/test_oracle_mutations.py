"""The pins have teeth: a plausible mistake planted in a copy of an oracle's source makes at
least one of its pins fail.
  - The operator's C oracle (a wrong scale index or layout stride, a wrong exponent bias, a
    dropped or misplaced term, a wrong sign, an off-by-one range, swapped nibbles): each mutant
    is built with the oracle's own compiler flags and run through test_oracle_pins.py in a
    child process (GMMFR_ORACLE_LIB points the oracle at it).
  - The routing and FFN oracles (numpy) and the operator oracle's argument marshalling
    (Python): the pins of test_route_oracle.py / test_ffn_oracle.py / test_oracle_pins.py run in
    a child process whose conftest swaps in the functions of the mutated source
    (GMMFR_ORACLE_PY_MUTANT)."""
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
    ("E2M1 subnormal step", "e == 0 ? 0.5 * m :", "e == 0 ? 1.0 * m :"),
    ("E2M1 exponent bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)"),
    ("E5M2 infinity read as NaN", "return s ? -INFINITY : INFINITY;", "return NAN;"),
    ("E8M0 NaN code read as a power of two", "if (code == 255) return NAN;", "if (code == 256) return NAN;"),
    ("per-expert scale stride", "e * Ks * a->N * 2 : 0;", "e * Ks * a->N : 0;"),
    ("transposed x2 read untransposed", "if (a->transpose_x2) return element_code(", "if (0) return element_code("),
    ("bias of expert 0 for every expert", "a->bias[e * N + n0 + j]", "a->bias[n0 + j]"),
    ("shared rows placed from row 0", "const int64_t r = a->shared_offset + i;", "const int64_t r = i;"),
    ("bad row index not flagged", "flags |= ORACLE_BAD_ROW_INDEX;", "flags |= 0;"),
    ("count past M not flagged", "if (g < 0 || g > a->M - s) flags |= ORACLE_BAD_GROUP_LIST;",
     "if (g < 0) flags |= ORACLE_BAD_GROUP_LIST;"),
    ("sampled path drops the logit", "v += lg * (acc + b);", "v += acc + b;"),
    ("sampled path drops the shared weight", "v += a->shared_weight * oracle_decode_bf16(",
     "v += oracle_decode_bf16("),
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


@pytest.fixture(scope="module")
def mutant_libs(tmp_path_factory):
    import oracle
    oracle.build()
    tmp = str(tmp_path_factory.mktemp("mutants"))
    return [_build(tmp, i, old, new) for i, (_, old, new) in enumerate(MUTANTS)]


def test_every_planted_mistake_fails_a_pin(mutant_libs):
    libs = mutant_libs
    with cf.ThreadPoolExecutor(min(8, os.cpu_count() or 1)) as ex:
        caught = list(ex.map(_pins_fail, libs))
    survivors = [m[0] for m, c in zip(MUTANTS, caught) if not c]
    assert not survivors, f"mutants no pin catches: {survivors}"


# (module, pins, name, text in the module's source (exactly once), replacement)
PY_MUTANTS = [
    ("oracle.route", "test_route_oracle.py", "invalid ids sorted first", "key = np.where(valid, flat, E)",
     "key = np.where(valid, flat, -1)"),
    ("oracle.route", "test_route_oracle.py", "ties in descending entry order",
     'perm = np.argsort(key, kind="stable").astype(np.int64)',
     'perm = (key.size - 1 - np.argsort(key[::-1], kind="stable")).astype(np.int64)'),
    ("oracle.route", "test_route_oracle.py", "group_list types swapped",
     "group_list = counts if group_list_type == 1 else np.cumsum(counts)",
     "group_list = np.cumsum(counts) if group_list_type == 1 else counts"),
    ("oracle.route", "test_route_oracle.py", "invalid ids counted", "np.bincount(flat[valid], minlength=E)",
     "np.bincount(np.clip(flat, 0, E - 1), minlength=E)"),
    ("oracle.route", "test_route_oracle.py", "rows not permuted", "src_row = perm // topk",
     "src_row = np.arange(perm.size) // topk"),
    ("oracle.route", "test_route_oracle.py", "logit not permuted", "else w[perm],", "else w,"),
    ("oracle.ffn", "test_ffn_oracle.py", "SiLU sign", "g / (1.0 + np.exp(-g))", "g / (1.0 + np.exp(g))"),
    ("oracle.ffn", "test_ffn_oracle.py", "gate and up swapped", "silu(gu[:, :I]) * gu[:, I:]",
     "silu(gu[:, I:]) * gu[:, :I]"),
    ("oracle.ffn", "test_ffn_oracle.py", "sw not cast to bf16", "sw = round_bf16(silu(gu[:, :I]) * gu[:, I:])",
     "sw = silu(gu[:, :I]) * gu[:, I:]"),
    ("oracle.ffn", "test_ffn_oracle.py", "result not cast to bf16", "res[s:t] = round_bf16(sw @ w2e)",
     "res[s:t] = sw @ w2e"),
    ("oracle.ffn", "test_ffn_oracle.py", "bf16 with 7 significant bits", "r = np.round(m * 256.0)",
     "r = np.round(m * 128.0) * 2"),
    ("oracle.ffn", "test_ffn_oracle.py", "ties away from zero", "r = np.round(m * 256.0)",
     "r = np.trunc(m * 256.0 + np.sign(m) * 0.5)"),
    ("oracle.ffn", "test_ffn_oracle.py", "w2 of expert 0 for every expert", "w2e = w2[e * I:(e + 1) * I]",
     "w2e = w2[0:I]"),
    ("oracle.ffn", "test_ffn_oracle.py", "expert range one row short", "s, t = int(cs[e]), int(cs[e + 1])",
     "s, t = int(cs[e]), int(cs[e + 1]) - (1 if cs[e + 1] > cs[e] else 0)"),
    ("oracle.ffn", "test_ffn_oracle.py", "error bound inflated", "absb[s:t] = np.abs(sw) @ np.abs(w2e)",
     "absb[s:t] = 10 * (np.abs(sw) @ np.abs(w2e))"),
    ("oracle.ffn", "test_ffn_oracle.py", "tolerance four bf16 steps", "return 2.0 ** -7 * np.abs(result)",
     "return 2.0 ** -5 * np.abs(result)"),
    ("oracle.ffn", "test_ffn_oracle.py", "tolerance without the sw term", "+ 1.1 * 2.0 ** -7 * absb",
     "+ 0.0 * absb"),
    ("oracle.route", "test_route_oracle.py", "scales gathered in token order", "pertoken_scale=xs[src_row],",
     "pertoken_scale=xs[np.sort(src_row)],"),
    ("oracle.route", "test_route_oracle.py", "bad ids not flagged", "flags=0 if bool(valid.all()) else BAD_EXPERT_ID,",
     "flags=0,"),
    # the operator oracle's argument marshalling (oracle/__init__.py)
    ("oracle", "test_oracle_pins.py", "transpose flag dropped", "transpose_x2=int(bool(transpose_x2))",
     "transpose_x2=0"),
    ("oracle", "test_oracle_pins.py", "per-expert scale flag dropped", "scale_per_expert=int(bool(scale_per_expert))",
     "scale_per_expert=0"),
    ("oracle", "test_oracle_pins.py", "shared weight fixed at 1", "shared_weight=float(shared_weight)",
     "shared_weight=1.0"),
    ("oracle", "test_oracle_pins.py", "group_list read as counts", "group_list_type=int(group_list_type)",
     "group_list_type=1"),
    ("oracle", "test_oracle_pins.py", "logit not passed", 'logit=ptr(k["logit"])', "logit=None"),
    ("oracle", "test_oracle_pins.py", "sampled rows and columns swapped",
     "rows.size, rows.ctypes.data_as(ctypes.c_void_p),\n                                     cols.ctypes",
     "rows.size, cols.ctypes.data_as(ctypes.c_void_p),\n                                     rows.ctypes"),
]


def _module_path(module):
    path = os.path.join(ROOT, *module.split("."))
    return os.path.join(path, "__init__.py") if os.path.isdir(path) else path + ".py"


def _py_pins_fail(tmp, i, module, pins, old, new):
    src_path = _module_path(module)
    src = open(src_path).read()
    assert src.count(old) == 1, old
    path = os.path.join(tmp, f"py{i}.py")
    open(path, "w").write(src.replace(old, new))
    env = dict(os.environ, GMMFR_ORACLE_PY_MUTANT=f"{module}={path}", OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", pins), "-x", "-q",
                        "-p", "no:cacheprovider"], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    return r.returncode == 1 and " failed" in r.stdout


def test_every_planted_mistake_in_the_numpy_oracles_fails_a_pin(tmp_path):
    with cf.ThreadPoolExecutor(min(8, os.cpu_count() or 1)) as ex:
        caught = list(ex.map(lambda a: _py_pins_fail(str(tmp_path), *a),
                             [(i, m[0], m[1], m[3], m[4]) for i, m in enumerate(PY_MUTANTS)]))
    survivors = [m[2] for m, c in zip(PY_MUTANTS, caught) if not c]
    assert not survivors, f"mutants no pin catches: {survivors}"
    # the unmodified sources pass their pins by the same route
    for module, pins in (("oracle.route", "test_route_oracle.py"), ("oracle.ffn", "test_ffn_oracle.py"),
                         ("oracle", "test_oracle_pins.py")):
        path = _module_path(module)
        env = dict(os.environ, GMMFR_ORACLE_PY_MUTANT=f"{module}={path}", OMP_NUM_THREADS="1")
        r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", pins), "-q",
                            "-p", "no:cacheprovider"], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout[-2000:]


def test_the_unmodified_source_passes_through_the_same_route(tmp_path):
    lib = _build(str(tmp_path), 0, "(int)code - 127", "(int)code - 127")
    env = dict(os.environ, GMMFR_ORACLE_LIB=lib, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-q",
                        "-p", "no:cacheprovider"], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]


# ----------------------------------------------------------------------------- the parity tolerance
# Mistakes whose effect the GPU parity comparison cannot see by construction: a doubled E5M2
# subnormal moves a result far less than the bound allows (1e-4 of the sum of |products|), and
# Inf / NaN decoding only shows on inputs holding those codes (pinned above, and by the NaN
# placement parity test).
_BELOW_TOLERANCE = {"E5M2 subnormal exponent", "E5M2 infinity read as NaN", "E8M0 NaN code read as a power of two"}


def _cases():
    """Small workloads of the GPU parity suite's kinds, with a bad row and a bad group_list."""
    import torch

    from moe_grouped_gemm_mxfp8_gb300 import workloads as W

    base = dict(name="t", batch=16, M=40, K=256, N=320, E=4, seed=11)
    kinds = [
        dict(rows="random", shared_rows=6, shared_offset=5, shared_weight=0.7, out_init="randn"),
        dict(transpose_x2=True, bias=True, rows="random"),
        dict(x1_dtype=W.E5M2, x2_dtype=W.E5M2, group_list_type=0, scale_lo=120, scale_hi=134),
        dict(scale_per_expert=True),
        dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1),
        dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, transpose_x2=True, K=352, N=200),
    ]
    out = []
    for kw in kinds:
        spec = W.Spec(**dict(base, **kw))
        out.append((spec, W.make_inputs(spec)))
    spec = W.Spec(**dict(base, rows="random"))
    inp = W.make_inputs(spec)
    inp["row_index"][3] = spec.batch                                   # a bad row
    out.append((spec, inp))
    spec = W.Spec(**dict(base, counts="explicit", explicit_counts=(10, 10, 10, 10)))
    inp = W.make_inputs(spec)
    inp["group_list"] = torch.tensor([12, 8, 10, 15], dtype=torch.int64)  # counts past M
    out.append((spec, inp))
    return out


def _mutant_runs(lib_path, p, rows, cols):
    import ctypes

    import numpy as np

    import oracle
    lib = ctypes.CDLL(lib_path)
    P = ctypes.POINTER(oracle._Args)
    vp = ctypes.c_void_p
    lib.oracle_gmmfr.argtypes = [P, vp, vp]
    lib.oracle_gmmfr_sampled.argtypes = [P, ctypes.c_int64, vp, vp, vp, vp]
    full = np.zeros((p.batch, p.N))
    absb = np.zeros((p.batch, p.N))
    flags = lib.oracle_gmmfr(ctypes.byref(p.args), full.ctypes.data_as(vp), absb.ctypes.data_as(vp))
    vals = np.zeros(rows.size)
    bnd = np.zeros(rows.size)
    sflags = lib.oracle_gmmfr_sampled(ctypes.byref(p.args), rows.size, rows.ctypes.data_as(vp),
                                      cols.ctypes.data_as(vp), vals.ctypes.data_as(vp), bnd.ctypes.data_as(vp))
    return full, flags, vals, sflags


def test_parity_tolerance_rejects_each_arithmetic_mistake(mutant_libs):
    """The GPU parity tests accept a result within oracle.tolerance of the oracle and with the
    same error flags.  Each planted mistake, if it were the kernel's, would fail that check on
    at least one small workload of the kinds the GPU suite runs (the GPU suite compares every
    element; mistakes planted in the oracle's per-element entry point are judged by that entry
    point's output)."""
    import numpy as np

    import oracle

    cases = []
    for spec, inp in _cases():
        p = oracle.problem_from_spec(spec, inp)
        ref, absb, flags = oracle.run(p)
        bound = oracle.tolerance(ref, absb)
        rr, cc = np.meshgrid(np.arange(spec.batch), np.arange(spec.N), indexing="ij")
        cases.append((p, ref, flags, bound, rr.ravel().astype(np.int64), cc.ravel().astype(np.int64)))
    unseen = []
    for (name, _, _), lib in zip(MUTANTS, mutant_libs):
        if name in _BELOW_TOLERANCE:
            continue
        seen = False
        for p, ref, flags, bound, rows, cols in cases:
            full, mflags, vals, sflags = _mutant_runs(lib, p, rows, cols)
            bad_full = mflags != flags or not np.all(np.abs(full - ref) <= bound)
            bad_sampled = sflags != flags or not np.all(np.abs(vals - ref.ravel()) <= bound.ravel())
            if bad_full or bad_sampled:
                seen = True
                break
        if not seen:
            unseen.append(name)
    assert not unseen, f"mistakes the parity tolerance accepts: {unseen}"
