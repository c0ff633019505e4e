"""GPU parity of the routing step (bit-exact against the oracle) and of
routing followed by the operator, against the oracle of both."""
import numpy as np
import pytest
import torch

import oracle
from oracle import route as R
from moe_grouped_gemm_mxfp8_gb300 import binding as B
from moe_grouped_gemm_mxfp8_gb300 import build as build_mod
from moe_grouped_gemm_mxfp8_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    oracle.build()
    B.load()


CASES = [
    dict(batch=5, topk=2, K=64, E=4),
    dict(batch=300, topk=3, K=200, E=7, invalid=11),           # K not a multiple of 16, bad ids
    dict(batch=512, topk=8, K=7168, E=256),                    # the large benchmark routing
    dict(batch=1000, topk=1, K=128, E=1),
    dict(batch=777, topk=6, K=512, E=1024, invalid=1),
    dict(batch=0, topk=4, K=128, E=8),
    dict(batch=2048, topk=4, K=8192, E=256),                   # 8192 entries: the largest single-launch case
    dict(batch=3001, topk=4, K=144, E=64, invalid=5),          # 12004 entries: the three-launch path
]


@pytest.mark.parametrize("kw", CASES, ids=[str(i) for i in range(len(CASES))])
@pytest.mark.parametrize("ids32", [False, True])
@pytest.mark.parametrize("glt", [0, 1])
def test_route_bit_exact(kw, ids32, glt):
    spec = W.RouteSpec("t", seed=kw["batch"] + kw["E"], **kw)
    inp = W.make_route_inputs(spec)
    ref = R.moe_route(inp["topk_ids"].numpy(), inp["topk_weights"].numpy(), inp["x"].numpy(),
                      inp["x_scale"].numpy(), spec.E, glt)
    ids = inp["topk_ids"].to(torch.int32) if ids32 else inp["topk_ids"]
    out, ws = B.route(ids.cuda(), inp["topk_weights"].cuda(), inp["x"].cuda(), inp["x_scale"].cuda(), spec.E, glt)
    bits = B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert bits == (B.DEV_BAD_EXPERT_ID if ref["flags"] else 0)
    for k in ("perm", "x1", "pertoken_scale", "group_list", "row_index", "logit"):
        got = out[k].cpu().numpy()
        assert np.array_equal(got.reshape(ref[k].shape).astype(ref[k].dtype), ref[k]), k


@pytest.mark.parametrize("run", [80, 1000])
def test_route_runs_of_equal_ids(run):
    """Expert ids in runs of equal values (80: runs that start and end inside warps of 32
    entries; 1000: most warps hold one id), with invalid ids in one run: warps whose 32 keys
    are equal are counted in one step, the others entry by entry."""
    batch, topk, E = 1500, 2, 6
    spec = W.RouteSpec("t", batch=batch, topk=topk, K=96, E=E, seed=run)
    inp = W.make_route_inputs(spec)
    flat = (np.arange(batch * topk) // run) % E
    flat[2 * run:3 * run] = E + 2  # the third run: invalid ids
    ids = torch.from_numpy(flat.reshape(batch, topk).astype(np.int64))
    ref = R.moe_route(ids.numpy(), inp["topk_weights"].numpy(), inp["x"].numpy(), inp["x_scale"].numpy(), E, 1)
    out, ws = B.route(ids.cuda(), inp["topk_weights"].cuda(), inp["x"].cuda(), inp["x_scale"].cuda(), E, 1)
    bits = B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert bits == B.DEV_BAD_EXPERT_ID and ref["flags"]
    for k in ("perm", "x1", "pertoken_scale", "group_list", "row_index", "logit"):
        got = out[k].cpu().numpy()
        assert np.array_equal(got.reshape(ref[k].shape).astype(ref[k].dtype), ref[k]), k


@pytest.mark.parametrize("kw", [CASES[1], CASES[2], CASES[4], CASES[5]], ids=["1", "2", "4", "5"])
def test_route_three_launch_path_bit_exact(kw, monkeypatch):
    """Below 8193 entries the library routes in one launch; the three-launch path
    (count, scan, scatter) gives the same bytes."""
    monkeypatch.setenv("GMMFR_ROUTE_SPLIT", "1")
    spec = W.RouteSpec("t", seed=kw["batch"] + kw["E"], **kw)
    inp = W.make_route_inputs(spec)
    ref = R.moe_route(inp["topk_ids"].numpy(), inp["topk_weights"].numpy(), inp["x"].numpy(),
                      inp["x_scale"].numpy(), spec.E, 1)
    out, ws = B.route(inp["topk_ids"].cuda(), inp["topk_weights"].cuda(), inp["x"].cuda(), inp["x_scale"].cuda(),
                      spec.E, 1)
    bits = B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert bits == (B.DEV_BAD_EXPERT_ID if ref["flags"] else 0)
    for k in ("perm", "x1", "pertoken_scale", "group_list", "row_index", "logit"):
        got = out[k].cpu().numpy()
        assert np.array_equal(got.reshape(ref[k].shape).astype(ref[k].dtype), ref[k]), k


def test_route_without_weights_writes_ones():
    spec = W.RouteSpec("t", batch=40, topk=3, K=64, E=5, seed=9)
    inp = W.make_route_inputs(spec)
    out, _ = B.route(inp["topk_ids"].cuda(), None, inp["x"].cuda(), inp["x_scale"].cuda(), spec.E)
    assert torch.all(out["logit"] == 1.0)


@pytest.mark.parametrize("det", [False, True])
def test_route_then_operator(det):
    """Routing on the GPU feeding the grouped GEMM on the GPU equals the oracle
    of the routing feeding the oracle of the operator (within the tolerance)."""
    batch, topk, K, N, E = 96, 4, 512, 384, 12
    rs = W.RouteSpec("t", batch=batch, topk=topk, K=K, E=E, seed=31)
    ri = W.make_route_inputs(rs)
    gspec = W.Spec("w", batch=batch, M=batch * topk, K=K, N=N, E=E, seed=32, shared_rows=batch, out_init="randn")
    gi = W.make_inputs(gspec)
    out, _ = B.route(ri["topk_ids"].cuda(), ri["topk_weights"].cuda(), ri["x"].cuda(), ri["x_scale"].cuda(), E)
    prob = B.problem_from_spec(gspec, deterministic=det)
    x2, sc = gi["x2"].cuda(), gi["scale"].cuda()
    prep = B.prepare_weights(prob, x2, sc)
    res = gi["out"].cuda().clone()
    d = dict(x1=out["x1"], pertoken_scale=out["pertoken_scale"], group_list=out["group_list"], logit=out["logit"],
             row_index=out["row_index"], shared_input=gi["shared_input"].cuda())
    B.run(prob, d, res, prepared=prep)
    got = res.cpu().numpy().astype(np.float64)
    r = R.moe_route(ri["topk_ids"].numpy(), ri["topk_weights"].numpy(), ri["x"].numpy(), ri["x_scale"].numpy(), E)
    p = oracle.Problem(M=batch * topk, K=K, N=N, E=E, batch=batch, x1=r["x1"], x2=gi["x2"], scale=gi["scale"],
                       pertoken_scale=r["pertoken_scale"], group_list=r["group_list"], row_index=r["row_index"],
                       out=gi["out"], logit=r["logit"], shared_input=gi["shared_input"])
    ref, absb, flags = oracle.run(p)
    bound = oracle.tolerance(ref, absb)
    assert flags == 0
    assert np.all(np.abs(got - ref) <= bound)


def test_operator_launched_right_after_routing():
    """The operator's GEMM is a programmatic dependent of the routing kernel (its launch
    overlaps the routing tail; it reads nothing before routing completes).  Weights are
    prepared first, so each operator call directly follows a routing call on the stream;
    three rounds with fresh routings, each checked against the oracles."""
    batch, topk, K, N, E = 128, 2, 1024, 512, 16
    gspec = W.Spec("w", batch=batch, M=batch * topk, K=K, N=N, E=E, seed=41, shared_rows=batch, out_init="randn")
    gi = W.make_inputs(gspec)
    prob = B.problem_from_spec(gspec)
    prep = B.prepare_weights(prob, gi["x2"].cuda(), gi["scale"].cuda())
    shared = gi["shared_input"].cuda()
    torch.cuda.synchronize()
    for rnd in range(3):
        rs = W.RouteSpec("t", batch=batch, topk=topk, K=K, E=E, seed=50 + rnd)
        ri = W.make_route_inputs(rs)
        dev = {k: v.cuda() for k, v in ri.items()}
        res = gi["out"].cuda().clone()
        torch.cuda.synchronize()
        out, _ = B.route(dev["topk_ids"], dev["topk_weights"], dev["x"], dev["x_scale"], E)
        d = dict(x1=out["x1"], pertoken_scale=out["pertoken_scale"], group_list=out["group_list"],
                 logit=out["logit"], row_index=out["row_index"], shared_input=shared)
        B.run(prob, d, res, prepared=prep)
        got = res.cpu().numpy().astype(np.float64)
        r = R.moe_route(ri["topk_ids"].numpy(), ri["topk_weights"].numpy(), ri["x"].numpy(), ri["x_scale"].numpy(), E)
        p = oracle.Problem(M=batch * topk, K=K, N=N, E=E, batch=batch, x1=r["x1"], x2=gi["x2"], scale=gi["scale"],
                           pertoken_scale=r["pertoken_scale"], group_list=r["group_list"], row_index=r["row_index"],
                           out=gi["out"], logit=r["logit"], shared_input=gi["shared_input"])
        ref, absb, flags = oracle.run(p)
        bound = oracle.tolerance(ref, absb)
        assert flags == 0
        assert np.all(np.abs(got - ref) <= bound), rnd
