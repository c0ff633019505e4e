"""Pins of the routing oracle (no GPU): a brute-force restatement of the stable
order, closed forms, and the composition routing -> grouped matmul finalize
routing == the direct top-k weighted sum of expert outputs."""
import numpy as np
import pytest
import torch

import oracle
from oracle import route as R
from moe_grouped_gemm_mxfp8_gb300 import workloads as W


def _brute_perm(ids, E):
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    order = []
    for e in range(E):
        order += [f for f, v in enumerate(flat) if v == e]
    order += [f for f, v in enumerate(flat) if not 0 <= v < E]
    return order


@pytest.mark.parametrize("batch,topk,E,invalid", [(5, 2, 4, 0), (9, 3, 5, 3), (16, 8, 8, 0), (7, 4, 3, 5), (1, 1, 1, 0)])
def test_order_matches_brute_force(batch, topk, E, invalid):
    spec = W.RouteSpec("t", batch=batch, topk=topk, K=64, E=E, invalid=invalid, seed=batch)
    inp = W.make_route_inputs(spec)
    r = R.moe_route(inp["topk_ids"].numpy(), inp["topk_weights"].numpy(), inp["x"].numpy(), inp["x_scale"].numpy(), E)
    assert r["perm"].tolist() == _brute_perm(inp["topk_ids"], E)
    flat = inp["topk_ids"].view(-1).tolist()
    assert r["group_list"].tolist() == [sum(1 for v in flat if v == e) for e in range(E)]
    assert r["flags"] == (R.BAD_EXPERT_ID if invalid else 0)
    f = r["perm"]
    assert np.array_equal(r["row_index"], f // topk)
    assert np.array_equal(r["x1"], inp["x"].numpy()[f // topk])
    assert np.array_equal(r["logit"], inp["topk_weights"].numpy().reshape(-1)[f])
    r0 = R.moe_route(inp["topk_ids"].numpy(), None, inp["x"].numpy(), inp["x_scale"].numpy(), E, group_list_type=0)
    assert r0["group_list"].tolist() == np.cumsum(r["group_list"]).tolist()
    assert np.all(r0["logit"] == 1.0)


def test_single_expert_keeps_token_order():
    ids = np.full((6, 3), 2)
    r = R.moe_route(ids, None, np.zeros((6, 32), np.uint8), np.zeros((6, 1, 2), np.uint8), 4)
    assert r["perm"].tolist() == list(range(18))
    assert r["group_list"].tolist() == [0, 0, 18, 0]


def test_routing_then_operator_equals_direct_topk_sum():
    """out[b, n] = sum_k w[b,k] * sum_kk A(b, kk) * B(id[b,k], kk, n): computed
    directly with torch-decoded float64 values, independently of any ordering."""
    batch, topk, K, N, E = 6, 3, 96, 20, 5
    rs = W.RouteSpec("t", batch=batch, topk=topk, K=K, E=E, seed=3)
    ri = W.make_route_inputs(rs)
    gspec = W.Spec("w", batch=batch, M=batch * topk, K=K, N=N, E=E, seed=4)
    gi = W.make_inputs(gspec)
    r = R.moe_route(ri["topk_ids"].numpy(), ri["topk_weights"].numpy(), ri["x"].numpy(), ri["x_scale"].numpy(), E)
    p = oracle.Problem(M=batch * topk, K=K, N=N, E=E, batch=batch, x1=r["x1"], x2=gi["x2"], scale=gi["scale"],
                       pertoken_scale=r["pertoken_scale"], group_list=r["group_list"], row_index=r["row_index"],
                       out=np.zeros((batch, N), np.float32), logit=r["logit"])
    out, _, flags = oracle.run(p)
    assert flags == 0
    f8 = lambda t: t.view(torch.float8_e4m3fn).to(torch.float64)
    e8 = lambda t: t.view(torch.float8_e8m0fnu).to(torch.float64)
    a = f8(ri["x"]) * e8(ri["x_scale"]).reshape(batch, -1).repeat_interleave(32, 1)[:, :K]
    b = f8(gi["x2"]) * e8(gi["scale"]).permute(0, 2, 1).reshape(-1, N).repeat_interleave(32, 0)[:K][None]
    ref = np.zeros((batch, N))
    for bb in range(batch):
        for k in range(topk):
            e = int(ri["topk_ids"][bb, k])
            ref[bb] += float(ri["topk_weights"][bb, k]) * (a[bb] @ b[0 if b.shape[0] == 1 else e]).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
