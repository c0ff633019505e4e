"""The allocation-free entry point, gmmfr_grouped_matmul_finalize_routing_static_scratch.

Callers that cannot allocate device memory (a host runtime whose pool owns the
device, or a serving loop where cudaMalloc is not allowed) get a form of the
operator that runs in the library's own static device scratch.  These tests call
it through the C ABI twice in a row and check each result against the
workspace-taking entry point, within the parity tolerance used by the other GPU
tests, and that the second call leaves the device's free memory and torch's
allocator as they were; they read the call's device error word back through its
own accessor, and check that a problem too large for the scratch is refused.

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


def _static_call(prob, d, out, prep, stream):
    B.gmmfr_grouped_matmul_finalize_routing_static_scratch(
        prob, B.view(d["x1"]), B.view(d["pertoken_scale"]), B.view(d["group_list"]), B.view(d["logit"]),
        B.view(d["row_index"]), B.view(d["shared_input"]), B.view(out), prep.data_ptr(), prep.numel(), stream)


# E2M1 tokens with E4M3 weights: the tokens are expanded to E4M3 inside the call, into the
# static array past its header
@pytest.mark.parametrize("deterministic,x1_dtype", [(False, W.E4M3), (True, W.E4M3), (False, W.E2M1)],
                         ids=["atomic", "deterministic", "e2m1_tokens"])
def test_static_scratch_matches_workspace_entry_point(deterministic, x1_dtype):
    spec = W.Spec("static scratch M300 K384 N320 E5", batch=64, M=300, K=384, N=320, E=5, rows="random",
                  counts="explicit", explicit_counts=(0, 150, 7, 120, 23), shared_rows=40, shared_offset=10,
                  shared_weight=0.7, out_init="randn", x1_dtype=x1_dtype, seed=23)
    inp = W.make_inputs(spec)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    prob = B.problem_from_spec(spec, deterministic)
    prep = B.prepare_weights(prob, d["x2"], d["scale"])
    stream = torch.cuda.current_stream().cuda_stream

    ref = d["out"].clone()
    B.run(prob, d, ref, prepared=prep)  # the entry point that takes a workspace
    ref = ref.cpu().numpy().astype(np.float64)

    o64, absb, _ = oracle.run(oracle.problem_from_spec(spec, inp))
    bound = oracle.tolerance(o64, absb)

    for i in range(2):
        out = d["out"].clone()
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        allocs0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        _static_call(prob, d, out, prep, stream)
        torch.cuda.synchronize()
        if i == 1:  # the call allocates nothing: device free memory and torch's allocator unchanged
            assert torch.cuda.mem_get_info()[0] == free0
            assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs0
        assert B.gmmfr_static_scratch_check_device_errors(stream) == 0
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= bound)
        assert np.all(np.abs(got - o64) <= bound)
        if deterministic:
            assert np.array_equal(got, ref)


def test_static_scratch_reports_device_errors():
    """A routed token whose row_index is outside [0, batch) is skipped and sets its bit in the
    static array's error word, which the accessor reads back; the next clean call clears it."""
    spec = W.Spec("static scratch bad row", batch=16, M=40, K=256, N=128, E=2, rows="random", seed=24)
    inp = W.make_inputs(spec)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    prob = B.problem_from_spec(spec)
    prep = B.prepare_weights(prob, d["x2"], d["scale"])
    stream = torch.cuda.current_stream().cuda_stream
    bad = dict(d, row_index=d["row_index"].clone())
    bad["row_index"][3] = spec.batch
    _static_call(prob, bad, d["out"].clone(), prep, stream)
    assert B.gmmfr_static_scratch_check_device_errors(stream) == B.DEV_BAD_ROW_INDEX
    _static_call(prob, d, d["out"].clone(), prep, stream)
    assert B.gmmfr_static_scratch_check_device_errors(stream) == 0


def test_static_scratch_refuses_oversized_problems():
    # Deterministic mode keeps one FP32 partial per (token, column): 4096 x 4096 x 4 B = 64 MiB,
    # beyond the 16 MiB scratch.  Every tensor pointer is NULL, so even a call that got past
    # the size check would be refused by host validation before anything is enqueued.
    big = B.make_problem(M=4096, K=7168, N=4096, E=256, batch=512, deterministic=True)
    assert B.gmmfr_workspace_size(big, True) > 16 << 20
    with pytest.raises(B.GmmfrError) as ei:
        B.gmmfr_grouped_matmul_finalize_routing_static_scratch(big, None, None, None, None, None, None, None, 256,
                                                               1 << 40)
    assert ei.value.status == B.ERR_WORKSPACE and "16 MiB" in str(ei.value)
    small = B.make_problem(M=16, K=128, N=128, E=1, batch=16)
    with pytest.raises(B.GmmfrError) as ei:
        B.gmmfr_grouped_matmul_finalize_routing_static_scratch(small, None, None, None, None, None, None, None, None,
                                                               0)
    assert ei.value.status == B.ERR_INVALID_ARG and "gmmfr_prepare_weights" in str(ei.value)
