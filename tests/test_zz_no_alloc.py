"""The allocation-free entry point, gmmfr_grouped_matmul_finalize_routing_static_scratch.

Callers that cannot allocate device memory (a host runtime whose pool owns the
device, or a serving loop where cudaMalloc is not allowed) get a form of the
operator that runs in the library's own static device scratch.  These tests call
it through the C ABI twice in a row and check each result against the
workspace-taking entry point, within the parity tolerance used by the other GPU
tests, and check that a problem too large for the scratch is refused.

This file is collected last on purpose: a run that stops at its first failure
has then already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
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


@pytest.mark.parametrize("deterministic", [False, True])
def test_static_scratch_matches_workspace_entry_point(deterministic):
    spec = W.Spec("static scratch M300 K384 N320 E5", batch=64, M=300, K=384, N=320, E=5, rows="random",
                  counts="explicit", explicit_counts=(0, 150, 7, 120, 23), shared_rows=40, shared_offset=10,
                  shared_weight=0.7, out_init="randn", seed=23)
    inp = W.make_inputs(spec)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    prob = B.problem_from_spec(spec, deterministic)
    prep = B.prepare_weights(prob, d["x2"], d["scale"])
    stream = torch.cuda.current_stream().cuda_stream

    ref = d["out"].clone()
    B.run(prob, d, ref, prepared=prep)  # the entry point that takes a workspace
    ref = ref.cpu().numpy().astype(np.float64)

    o64, absb, _ = oracle.run(oracle.problem_from_spec(spec, inp))
    init = inp["out"].numpy().astype(np.float64)
    sh = np.zeros_like(init)
    sh[10:50] = 0.7 * inp["shared_input"].to(torch.float64).numpy()
    bound = oracle.tolerance(o64, absb, init, sh)

    for _ in range(2):
        out = d["out"].clone()
        B.gmmfr_grouped_matmul_finalize_routing_static_scratch(
            prob, d["x1"].data_ptr(), d["pertoken_scale"].data_ptr(), d["group_list"].data_ptr(),
            d["logit"].data_ptr(), d["row_index"].data_ptr(), d["shared_input"].data_ptr(), out.data_ptr(),
            prep.data_ptr(), stream)
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= bound)
        assert np.all(np.abs(got - o64) <= bound)
        if deterministic:
            assert np.array_equal(got, ref)


def test_static_scratch_refuses_oversized_problems():
    # Deterministic mode keeps one FP32 partial per (token, column): 4096 x 4096 x 4 B = 64 MiB,
    # beyond the 16 MiB scratch.  Every tensor pointer is NULL, so even a call that got past
    # the size check would be refused by host validation before anything is enqueued.
    big = B.make_problem(M=4096, K=7168, N=4096, E=256, batch=512, deterministic=True)
    assert B.gmmfr_workspace_size(big, True) > 16 << 20
    with pytest.raises(B.GmmfrError) as ei:
        B.gmmfr_grouped_matmul_finalize_routing_static_scratch(big, None, None, None, None, None, None, None, 256)
    assert ei.value.status == B.ERR_WORKSPACE and "16 MiB" in str(ei.value)
    small = B.make_problem(M=16, K=128, N=128, E=1, batch=16)
    with pytest.raises(B.GmmfrError) as ei:
        B.gmmfr_grouped_matmul_finalize_routing_static_scratch(small, None, None, None, None, None, None, None, None)
    assert ei.value.status == B.ERR_INVALID_ARG and "gmmfr_prepare_weights" in str(ei.value)
