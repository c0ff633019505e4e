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
    (dict(K=5121, x1_format=2), B.ERR_INVALID_ARG, "even K"),
    (dict(K=5121, x2_format=2, transpose_x2=1), B.ERR_INVALID_ARG, "even K"),
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
        B.gmmfr_grouped_matmul_finalize_routing(p, *[None] * 10, 256, 1 << 40, 256, 1 << 30)
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


# ----------------------------------------------------------------------------- tensor views
# Every call below fails on the host before anything is enqueued: the addresses are not real
# device memory, and a call that passes every view check still stops at the workspace check
# (a 16-byte workspace), so no test here launches a kernel.
def _views(p, **over):
    """Views of the operator's tensors for problem p, at a fake 256-byte-aligned address."""
    Ks = -(-p.K // 64)
    v = dict(x1=B.raw_view(256, B.DT_E4M3, (p.M, p.K)), x2=None, scale=None,
             pts=B.raw_view(256, B.DT_U8, (p.M, Ks, 2)), gl=B.raw_view(256, B.DT_I64, (p.E,)),
             logit=B.raw_view(256, B.DT_F32, (p.M,)), rows=B.raw_view(256, B.DT_I64, (p.M,)),
             shared=B.raw_view(256, B.DT_BF16, (p.shared_rows, p.N)), bias=None,
             out=B.raw_view(256, B.DT_F32, (p.batch, p.N)))
    v.update(over)
    return v


def _call(p, v, prepared=256, prepared_bytes=1 << 40, ws=256, ws_bytes=16):
    B.gmmfr_grouped_matmul_finalize_routing(p, v["x1"], v["x2"], v["scale"], v["pts"], v["gl"], v["logit"],
                                            v["rows"], v["shared"], v["bias"], v["out"], prepared, prepared_bytes,
                                            ws, ws_bytes)


def test_valid_views_reach_the_workspace_check(lib):
    p = _ok_problem()
    with pytest.raises(B.GmmfrError, match="workspace has 16 bytes") as ei:
        _call(p, _views(p))
    assert ei.value.status == B.ERR_WORKSPACE
    # typed FP8 and E8M0 codes, int32 rows with row_index_type int32, a bias, raw weights
    p32 = _ok_problem(row_index_type=B.INDEX_I32)
    Ks = -(-p32.K // 64)
    v = _views(p32, rows=B.raw_view(256, B.DT_I32, (p32.M,)), pts=B.raw_view(256, B.DT_E8M0, (p32.M, Ks, 2)),
               bias=B.raw_view(256, B.DT_BF16, (p32.E, p32.N)),
               x2=B.raw_view(256, B.DT_E4M3, (p32.E, p32.K, p32.N)), scale=B.raw_view(256, B.DT_U8, (Ks, p32.N, 2)))
    with pytest.raises(B.GmmfrError, match="workspace has 16 bytes"):
        _call(p32, v, prepared=None, prepared_bytes=0)
    # packed E2M1 tokens: [M, K/2] bytes
    p4 = _ok_problem(x1_format=2, x2_format=2)
    with pytest.raises(B.GmmfrError, match="workspace has 16 bytes"):
        _call(p4, _views(p4, x1=B.raw_view(256, B.DT_E2M1X2, (p4.M, p4.K // 2))))


def _bad(p):
    Ks = -(-p.K // 64)
    M, K, N, E, batch, R = p.M, p.K, p.N, p.E, p.batch, p.shared_rows
    return [
        ("x1 missing", dict(x1=None), "x1 is required"),
        ("x1 dtype", dict(x1=B.raw_view(256, B.DT_E5M2, (M, K))), "x1: element type E5M2"),
        ("x1 float", dict(x1=B.raw_view(256, B.DT_F32, (M, K))), "x1: element type F32"),
        ("x1 shape", dict(x1=B.raw_view(256, B.DT_U8, (M, K + 16))), "x1: shape"),
        ("x1 rank", dict(x1=B.raw_view(256, B.DT_U8, (M * K,))), "x1: rank 1, expected 2"),
        ("x1 strides", dict(x1=B.raw_view(256, B.DT_U8, (M, K), (2 * K, 1))), "dense row-major"),
        ("x1 column-major", dict(x1=B.raw_view(256, B.DT_U8, (M, K), (1, M))), "dense row-major"),
        ("x1 data", dict(x1=B.raw_view(None, B.DT_U8, (M, K))), "x1: data is NULL"),
        ("x1 misaligned", dict(x1=B.raw_view(264, B.DT_U8, (M, K))), "x1 must be 16-byte aligned"),
        ("pertoken_scale shape", dict(pts=B.raw_view(256, B.DT_U8, (M, Ks + 1, 2))), "pertoken_scale: shape"),
        ("pertoken_scale dtype", dict(pts=B.raw_view(256, B.DT_F32, (M, Ks, 2))), "pertoken_scale: element type"),
        ("group_list dtype", dict(gl=B.raw_view(256, B.DT_I32, (E,))), "group_list: element type I32"),
        ("group_list shape", dict(gl=B.raw_view(256, B.DT_I64, (E + 1,))), "group_list: shape"),
        ("group_list missing", dict(gl=None), "group_list is required"),
        ("logit dtype", dict(logit=B.raw_view(256, B.DT_BF16, (M,))), "logit: element type BF16"),
        ("logit shape", dict(logit=B.raw_view(256, B.DT_F32, (M - 1,))), "logit: shape"),
        ("row_index dtype", dict(rows=B.raw_view(256, B.DT_I32, (M,))), "row_index: element type I32"),
        ("row_index missing", dict(rows=None), "row_index is required"),
        ("shared_input missing", dict(shared=None), "shared_input is required"),
        ("shared_input shape", dict(shared=B.raw_view(256, B.DT_BF16, (R + 1, N))), "shared_input: shape"),
        ("shared_input dtype", dict(shared=B.raw_view(256, B.DT_F32, (R, N))), "shared_input: element type"),
        ("bias shape", dict(bias=B.raw_view(256, B.DT_BF16, (E, N + 1))), "bias: shape"),
        ("out dtype", dict(out=B.raw_view(256, B.DT_BF16, (batch, N))), "out: element type BF16"),
        ("out shape", dict(out=B.raw_view(256, B.DT_F32, (batch + 1, N))), "out: shape"),
        ("out missing", dict(out=None), "out is required"),
        ("x2 transposed layout", dict(x2=B.raw_view(256, B.DT_U8, (E, N, K)),
                                      scale=B.raw_view(256, B.DT_U8, (Ks, N, 2))), "x2: shape"),
        ("scale of the other layout", dict(x2=B.raw_view(256, B.DT_U8, (E, K, N)),
                                           scale=B.raw_view(256, B.DT_U8, (N, Ks, 2))), "scale: shape"),
    ]


@pytest.mark.parametrize("i", range(len(_bad(_ok_problem()))), ids=[b[0] for b in _bad(_ok_problem())])
def test_views_that_do_not_match_the_problem_are_refused(lib, i):
    p = _ok_problem()
    name, over, msg = _bad(p)[i]
    prepared = None if "x2" in over else 256
    with pytest.raises(B.GmmfrError) as ei:
        _call(p, _views(p, **over), prepared=prepared)
    assert ei.value.status == B.ERR_INVALID_ARG and msg in str(ei.value), str(ei.value)


def test_weight_views_and_buffers(lib):
    p = _ok_problem()
    Ks = -(-p.K // 64)
    # no prepared weights and no raw weights
    with pytest.raises(B.GmmfrError, match="x2 is required"):
        _call(p, _views(p), prepared=None, prepared_bytes=0)
    # a prepared buffer smaller than the problem's prepared weights
    need = B.gmmfr_prepared_weights_size(p)
    with pytest.raises(B.GmmfrError, match="prepared buffer has") as ei:
        _call(p, _views(p), prepared_bytes=need - 1)
    assert ei.value.status == B.ERR_WORKSPACE
    # the 4-D per-expert scale form
    pe = _ok_problem(scale_per_expert=1)
    v = _views(pe, x2=B.raw_view(256, B.DT_U8, (pe.E, pe.K, pe.N)), scale=B.raw_view(256, B.DT_U8, (Ks, pe.N, 2)))
    with pytest.raises(B.GmmfrError, match="scale: rank 3, expected 4"):
        _call(pe, v, prepared=None, prepared_bytes=0)
    # weight preparation checks its views the same way, then the buffer size (before any launch)
    x2 = B.raw_view(256, B.DT_U8, (p.E, p.K, p.N))
    sc = B.raw_view(256, B.DT_E8M0, (Ks, p.N, 2))
    with pytest.raises(B.GmmfrError, match="x2: shape"):
        B.gmmfr_prepare_weights(p, B.raw_view(256, B.DT_U8, (p.E, p.K, p.N - 1)), sc, 256, 1 << 40)
    with pytest.raises(B.GmmfrError, match="scale: element type F32"):
        B.gmmfr_prepare_weights(p, x2, B.raw_view(256, B.DT_F32, (Ks, p.N, 2)), 256, 1 << 40)
    with pytest.raises(B.GmmfrError, match="prepared buffer has"):
        B.gmmfr_prepare_weights(p, x2, sc, 256, need - 1)


@pytest.mark.parametrize("args,msg", [
    (dict(ws=None), "workspace is NULL"),
    (dict(ws=264, ws_bytes=1 << 40), "256-byte aligned"),
    (dict(ws_bytes=1024), "workspace has 1024 bytes"),
])
def test_bad_workspace_is_rejected_on_the_host(lib, args, msg):
    p = _ok_problem()
    with pytest.raises(B.GmmfrError) as ei:
        _call(p, _views(p), **args)
    assert msg in str(ei.value) and ei.value.status == B.ERR_WORKSPACE


def test_empty_problems_are_no_ops(lib):
    # N = 0 (aclnn: "x2 supports an empty tensor with N = 0"): nothing to enqueue, no tensor needed
    B.gmmfr_grouped_matmul_finalize_routing(_ok_problem(N=0), *[None] * 10, None, 0, None, 0)


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


def test_any_k_adds_the_padded_token_copy(lib):
    """K % 16 != 0 is accepted: the workspace grows by M * K rounded up to 16 for the copy of
    x1 at a 16-byte pitch (E2M1 tokens are expanded in the same copy)."""
    for K in (1, 40, 72, 200, 5128 + 3):
        p = _ok_problem(K=K)
        assert B.gmmfr_workspace_size(p, True) == 4096 + -(-(p.M * (-(-K // 16) * 16)) // 256) * 256
    p4 = _ok_problem(K=40, x1_format=2)
    assert B.gmmfr_workspace_size(p4, True) == 4096 + -(-(p4.M * 48) // 256) * 256
    # x1 need not be 16-byte aligned when it is copied first: the call passes host checks
    # up to the workspace check
    p = _ok_problem(K=40)
    with pytest.raises(B.GmmfrError, match="workspace has"):
        _call(p, _views(p, x1=B.raw_view(264, B.DT_U8, (p.M, p.K))))


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
