"""GPU parity of the grouped SwiGLU FFN (BF16, two tcgen05 kind::f16 grouped
GEMMs) against its oracle; tolerance per element from oracle/ffn.tolerance."""
import numpy as np
import pytest
import torch

from oracle import ffn as F
from moe_grouped_gemm_mxfp8_gb300 import binding as B
from moe_grouped_gemm_mxfp8_gb300 import build as build_mod
from moe_grouped_gemm_mxfp8_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    B.load()


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _check(spec, inp, extra_rows=0):
    d = {k: v.cuda() for k, v in inp.items()}
    N = d["sorted_tokens"].shape[0] + extra_rows
    x = torch.cat([d["sorted_tokens"], torch.ones((extra_rows, spec.H), dtype=torch.bfloat16, device="cuda")])
    prep = B.ffn_prepare(spec.H, spec.I, spec.E, d["w13_flat"], d["w2_flat"])
    init = torch.full((N, spec.H), 3.0, dtype=torch.bfloat16, device="cuda")  # rows outside the groups keep this
    res, ws = B.ffn(x, prep, d["expert_cumsum"], spec.H, spec.I, spec.E, result=init.clone())
    bits = B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    ref = F.grouped_swiglu_ffn(_bits(x), _bits(inp["w13_flat"]), _bits(inp["w2_flat"]), inp["expert_cumsum"].numpy(),
                               spec.H, spec.I, result_init=_bits(init))
    got = res.float().cpu().numpy().astype(np.float64)
    tol = F.tolerance(ref["result"], ref["absb"])
    err = np.abs(got - ref["result"])
    assert np.all(err <= tol), f"max err/tol {(err / tol).max():.3g}"
    assert bits == 0
    return got, ref


CASES = {
    "writeup_test": W.ffn_config("test"),
    "small": W.FfnSpec("s", H=128, I=64, E=3, counts=(5, 0, 9), scale=0.3, seed=1),
    "ragged_dims": W.FfnSpec("r", H=200, I=72, E=4, counts=(17, 33, 0, 70), scale=0.3, seed=2),
    "wide_groups": W.FfnSpec("w", H=256, I=128, E=3, counts=(129, 300, 64), scale=0.1, seed=3),
    "many_experts": W.FfnSpec("m", H=256, I=128, E=300, counts=tuple((i * 7) % 13 for i in range(300)), scale=0.2, seed=4),
}


@pytest.mark.parametrize("name", list(CASES))
def test_ffn_parity(name):
    spec = CASES[name]
    _check(spec, W.make_ffn_inputs(spec))


def test_rows_past_the_groups_are_untouched_and_deterministic():
    spec = CASES["small"]
    inp = W.make_ffn_inputs(spec)
    got, _ = _check(spec, inp, extra_rows=5)
    assert np.all(got[-5:] == 3.0)
    d = {k: v.cuda() for k, v in inp.items()}
    prep = B.ffn_prepare(spec.H, spec.I, spec.E, d["w13_flat"], d["w2_flat"])
    a, _ = B.ffn(d["sorted_tokens"], prep, d["expert_cumsum"], spec.H, spec.I, spec.E)
    b, _ = B.ffn(d["sorted_tokens"], prep, d["expert_cumsum"], spec.H, spec.I, spec.E)
    assert torch.equal(a, b)


def test_invalid_cumsum_sets_error_bit():
    spec = CASES["small"]
    inp = W.make_ffn_inputs(spec)
    d = {k: v.cuda() for k, v in inp.items()}
    d["expert_cumsum"] = torch.tensor([0, 9, 4, 14], dtype=torch.int32, device="cuda")  # decreasing
    prep = B.ffn_prepare(spec.H, spec.I, spec.E, d["w13_flat"], d["w2_flat"])
    _, ws = B.ffn(d["sorted_tokens"], prep, d["expert_cumsum"], spec.H, spec.I, spec.E)
    assert B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) & B.DEV_BAD_GROUP_LIST


def test_model_shape_full():
    """The benchmarked LLaDA2.0-mini shape (H 2048, I 512, E 256, 4096 routed tokens; LLaDA2
    grouped-GEMM write-up sections 3.2-3.3), with the weights drawn as the benchmark draws
    them (seeded CUDA generator): every result element against the oracle."""
    spec = W.ffn_config("model")
    inp = {k: v.cpu() for k, v in W.make_ffn_inputs(spec, weights_device="cuda").items()}
    torch.cuda.empty_cache()
    _check(spec, inp)
