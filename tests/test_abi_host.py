"""Host-side checks of the C ABI (no GPU): the library builds for sm_103a,
exports every entry point include/gmmfr.h declares, validates arguments before
any CUDA call, and the binding refuses to run without the library."""
import ctypes
import os
import re

import pytest

from moe_grouped_gemm_mxfp8_gb300 import binding as B
from moe_grouped_gemm_mxfp8_gb300 import build as build_mod
from moe_grouped_gemm_mxfp8_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(gmmfr_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_entry_point(lib):
    declared = _declared_functions()
    assert declared == set(B.ENTRY_POINTS)
    for name in declared:
        assert hasattr(lib, name), name
    # nothing but the C ABI is exported
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert {n for n in exported if n.startswith("gmmfr_")} == declared


def test_problem_struct_matches_header(lib):
    # sizeof(gmmfr_problem): 5 int64 + 6 int32 + 2 int64 + float + uint32 + int64
    assert ctypes.sizeof(B.Problem) == 5 * 8 + 6 * 4 + 2 * 8 + 4 + 4 + 8


def _ok_problem(**kw):
    base = dict(M=128, K=5120, N=4096, E=8, batch=64, shared_rows=64)
    base.update(kw)
    return B.make_problem(**base)


BAD = [
    (dict(E=0), B.ERR_INVALID_ARG, "E=0"),
    (dict(E=1025), B.ERR_INVALID_ARG, "E=1025"),
    (dict(M=-1), B.ERR_INVALID_ARG, "M=-1"),
    (dict(K=0), B.ERR_INVALID_ARG, "K=0"),
    (dict(N=-5), B.ERR_INVALID_ARG, "N=-5"),
    (dict(batch=-1, shared_rows=0), B.ERR_INVALID_ARG, "batch=-1"),
    (dict(x1_format=3), B.ERR_INVALID_ARG, "x1_format"),
    (dict(x2_format=2, N=63), B.ERR_INVALID_ARG, "even N"),
    (dict(x2_format=7), B.ERR_INVALID_ARG, "x2_format"),
    (dict(group_list_type=2), B.ERR_INVALID_ARG, "group_list_type"),
    (dict(row_index_type=5), B.ERR_INVALID_ARG, "row_index_type"),
    (dict(shared_offset=-1), B.ERR_INVALID_ARG, "negative"),
    (dict(shared_offset=1), B.ERR_INVALID_ARG, "exceeds batch"),
    (dict(shared_rows=65), B.ERR_INVALID_ARG, "exceeds batch"),
    (dict(K=5128), B.ERR_UNSUPPORTED, "K % 16"),
    (dict(expected_tokens_per_expert=-1), B.ERR_INVALID_ARG, "expected_tokens_per_expert"),
]


@pytest.mark.parametrize("kw,status,msg", BAD, ids=[b[2] for b in BAD])
def test_invalid_problems_are_rejected_on_the_host(lib, kw, status, msg):
    p = _ok_problem(**kw)
    with pytest.raises(B.GmmfrError) as ei:
        B.gmmfr_workspace_size(p, True)
    assert ei.value.status == status and msg in str(ei.value)
    # the operator itself rejects the same problem before enqueuing anything
    with pytest.raises(B.GmmfrError) as ei:
        B.gmmfr_grouped_matmul_finalize_routing(p, 16, None, None, 16, 16, None, 16, 16, None, 16, 16, 256, 1 << 30)
    assert ei.value.status == status


def test_flags_and_transpose_x1_like_inputs_are_rejected(lib):
    p = _ok_problem()
    p.flags = 6
    with pytest.raises(B.GmmfrError, match="flag"):
        B.gmmfr_workspace_size(p, True)
    p = _ok_problem()
    p.transpose_x2 = 3
    with pytest.raises(B.GmmfrError, match="transpose_x2"):
        B.gmmfr_workspace_size(p, True)


@pytest.mark.parametrize("args,msg", [
    (dict(x1=None), "x1, pertoken_scale and row_index"),
    (dict(gl=None), "group_list is NULL"),
    (dict(out=None), "out is NULL"),
    (dict(shared=None), "shared_input is NULL"),
    (dict(prepared=None), "either prepared or both x2 and scale"),
    (dict(x1=24), "x1 must be 16-byte aligned"),
    (dict(ws=None), "workspace is NULL"),
    (dict(ws=264), "256-byte aligned"),
    (dict(ws_bytes=1024), "workspace has 1024 bytes"),
])
def test_bad_pointers_are_rejected_on_the_host(lib, args, msg):
    p = _ok_problem()
    a = dict(x1=256, pts=256, gl=256, logit=256, rows=256, shared=256, out=256, prepared=256, ws=256,
             ws_bytes=1 << 40)
    a.update(args)
    with pytest.raises(B.GmmfrError) as ei:
        B.gmmfr_grouped_matmul_finalize_routing(p, a["x1"], None, None, a["pts"], a["gl"], a["logit"], a["rows"],
                                                a["shared"], None, a["out"], a["prepared"], a["ws"], a["ws_bytes"])
    assert msg in str(ei.value)
    assert ei.value.status in (B.ERR_INVALID_ARG, B.ERR_WORKSPACE)


def test_empty_problems_are_no_ops(lib):
    # N = 0 (aclnn: "x2 supports an empty tensor with N = 0"): nothing to enqueue
    B.gmmfr_grouped_matmul_finalize_routing(_ok_problem(N=0), None, None, None, None, 256, None, None, None,
                                            None, None, None, None, 0)


def test_sizes_follow_the_tiling(lib):
    for i in range(1, 6):
        s = W.config(i)
        p = B.problem_from_spec(s)
        nt, kb = -(-s.N // 128), -(-s.K // 128)
        assert B.gmmfr_prepared_weights_size(p) == s.E * nt * kb * 16896
        with_prep = B.gmmfr_workspace_size(p, True)
        without = B.gmmfr_workspace_size(p, False)
        assert without - with_prep >= s.E * nt * kb * 16896
        pd = B.problem_from_spec(s, deterministic=True)
        assert B.gmmfr_workspace_size(pd, True) >= with_prep + 4 * s.M * s.N


def test_e2m1_sizes_and_parity_rules(lib):
    """MXFP4: an odd N is allowed when x2 is transposed (packed along K).  E2M1 tokens
    and weights with K % 32 == 0 stay packed: tiles of 256 K elements (17408 bytes with
    their eight scales per row) and no token expansion.  Otherwise E2M1 tokens add M*K
    bytes of workspace for their E4M3 expansion and the weights become the FP8 tiles."""
    base = _ok_problem()
    n8 = B.gmmfr_workspace_size(base, True)
    p4 = _ok_problem(x1_format=2, x2_format=2)
    assert B.gmmfr_workspace_size(p4, True) == n8
    assert B.gmmfr_prepared_weights_size(p4) == p4.E * (-(-p4.N // 128)) * (-(-p4.K // 256)) * 17408
    assert B.gmmfr_workspace_size(p4, False) == n8 + B.gmmfr_prepared_weights_size(p4)
    for kw in (dict(x1_format=2, x2_format=0), dict(x1_format=2, x2_format=2, K=5120 + 16)):
        pm = _ok_problem(**kw)
        p8 = _ok_problem(K=pm.K)
        assert B.gmmfr_workspace_size(pm, True) >= B.gmmfr_workspace_size(p8, True) + pm.M * pm.K
        assert B.gmmfr_prepared_weights_size(pm) == B.gmmfr_prepared_weights_size(p8)
    p_w = _ok_problem(x2_format=2)  # FP8 tokens, E2M1 weights: FP8 tiles, no token workspace
    assert B.gmmfr_workspace_size(p_w, True) == n8
    assert B.gmmfr_prepared_weights_size(p_w) == B.gmmfr_prepared_weights_size(base)
    B.gmmfr_workspace_size(_ok_problem(x2_format=2, N=63, transpose_x2=1), True)
    B.gmmfr_workspace_size(_ok_problem(x1_format=2, N=63), True)


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        B.load(str(tmp_path / "missing.so"))


@pytest.mark.parametrize("kw,msg", [
    (dict(E=0), "out of range"), (dict(E=1025), "out of range"), (dict(topk=0), "out of range"),
    (dict(batch=-1), "out of range"), (dict(K=0), "out of range"), (dict(ids_type=3), "ids_type"),
    (dict(group_list_type=2), "group_list_type"),
])
def test_route_problem_validation(lib, kw, msg):
    base = dict(batch=8, topk=2, K=128, E=4, ids_type=0, group_list_type=1)
    base.update(kw)
    rp = B.RouteProblem(**base)
    with pytest.raises(B.GmmfrError, match=msg):
        B.gmmfr_moe_route_workspace_size(rp)
    with pytest.raises(B.GmmfrError):
        B.gmmfr_moe_route(rp, None, None, None, None, None, None, None, None, None, None, None, 0)


def test_route_rejects_missing_buffers(lib):
    rp = B.RouteProblem(batch=8, topk=2, K=128, E=4, ids_type=0, group_list_type=1)
    n = B.gmmfr_moe_route_workspace_size(rp)
    assert n >= 4096 + 16 * 4
    with pytest.raises(B.GmmfrError, match="must be non-NULL"):
        B.gmmfr_moe_route(rp, None, None, None, None, None, None, 256, None, None, None, 256, n)
    with pytest.raises(B.GmmfrError, match="workspace has"):
        B.gmmfr_moe_route(rp, 256, None, 256, 256, 256, 256, 256, 256, None, None, 256, 16)


@pytest.mark.parametrize("kw", [dict(H=100), dict(I=4), dict(E=0), dict(N=-1), dict(E=2000)])
def test_ffn_problem_validation(lib, kw):
    base = dict(N=16, H=128, I=64, E=4)
    base.update(kw)
    fp = B.FfnProblem(**base)
    with pytest.raises(B.GmmfrError, match="out of range"):
        B.gmmfr_ffn_workspace_size(fp)
    with pytest.raises(B.GmmfrError):
        B.gmmfr_llada2_moe_grouped_gemm(fp, None, None, None, None, None, 0)


def test_ffn_sizes(lib):
    fp = B.FfnProblem(N=4096, H=2048, I=512, E=256)
    assert B.gmmfr_ffn_prepared_weights_size(fp) == 256 * (8 * 32 + 16 * 8) * 16384
    assert B.gmmfr_ffn_workspace_size(fp) == 4096 + 4096 * 512 * 2
