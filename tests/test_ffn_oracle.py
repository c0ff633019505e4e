"""Pins of the grouped SwiGLU FFN oracle (no GPU)."""
import math

import numpy as np
import pytest
import torch

from oracle import ffn as F
from moe_grouped_gemm_mxfp8_gb300 import workloads as W


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000).astype(np.float32) * np.exp2(rng.integers(-20, 20, 20000)).astype(np.float32)
    # exact ties: a bf16 value plus half of its step
    base = rng.standard_normal(2000).astype(np.float32)
    b = torch.from_numpy(base).to(torch.bfloat16).to(torch.float32).numpy()
    ties = (b.view(np.uint32) + np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.round_bf16(x.astype(np.float64)), ref)
    assert np.array_equal(F.bf16_to_f64(F.f64_to_bf16_bits(ref)), ref)


def test_silu_anchor_values():
    assert F.silu(np.array(0.0)) == 0.0
    assert abs(F.silu(np.array(1.0)) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(F.silu(np.array(30.0)) - 30.0) < 1e-10
    assert abs(F.silu(np.array(-30.0))) < 1e-10
    g = np.linspace(-8, 8, 101)
    assert np.allclose(F.silu(g), torch.nn.functional.silu(torch.from_numpy(g)).numpy(), rtol=1e-15, atol=1e-18)


def test_closed_form_one_hot():
    """x = unit vector e_0, w13 row 0 = (a | b), w2 = identity on the first I
    columns: result[:, :I] = bf16(SiLU(a) * b) exactly, the rest zero."""
    H, I, E = 64, 32, 1
    x = np.zeros((3, H))
    x[:, 0] = 1.0
    a = np.linspace(-3, 3, I)
    b = np.linspace(0.5, 2, I)
    w13 = np.zeros((H, 2 * I))
    w13[0, :I], w13[0, I:] = a, b
    w2 = np.zeros((I, H))
    w2[np.arange(I), np.arange(I)] = 1.0
    bits = lambda v: F.f64_to_bf16_bits(v)
    r = F.grouped_swiglu_ffn(bits(x), bits(w13), bits(w2), np.array([0, 3]), H, I)
    ga, gb = F.bf16_to_f64(bits(a)), F.bf16_to_f64(bits(b))
    exp = F.round_bf16(ga / (1 + np.exp(-ga)) * gb)
    assert np.array_equal(r["result"][:, :I], np.tile(exp, (3, 1)))
    assert np.all(r["result"][:, I:] == 0)
    # absb = |sw| @ |w2|: here |sw| on the first I columns, 0 beyond
    assert np.array_equal(r["absb"][:, :I], np.tile(np.abs(exp), (3, 1)))
    assert np.all(r["absb"][:, I:] == 0)


def test_tolerance_admits_one_bf16_step():
    """With no sw term, the bound on a bf16 result r (|r| >= 1, where the 1e-7 floor is
    negligible) is at least the gap to the next bf16 value above |r| and less than twice it
    (two values a rounding apart land on adjacent bf16 values; a looser bound would hide a
    wrong rounding)."""
    rng = np.random.default_rng(3)
    mant = 1.0 + rng.random(5000)
    r = torch.from_numpy(np.where(rng.random(5000) < 0.5, -1, 1) * mant * np.exp2(rng.integers(0, 30, 5000)))
    r = r.to(torch.bfloat16)
    mag = r.abs()
    up = (mag.view(torch.int16) + 1).view(torch.bfloat16).to(torch.float64).numpy()
    step = up - mag.to(torch.float64).numpy()
    tol = F.tolerance(r.to(torch.float64).numpy(), np.zeros(r.numel()))
    assert np.all(tol >= step) and np.all(tol < 2 * step)


def test_both_bf16_casts_match_torch():
    """sw = bf16(SiLU(gate) * up) and result = bf16(sw @ w2_e), each cast checked against torch's
    own float64 -> bfloat16 conversion (the intermediate and the output are BF16, LLaDA2.0-mini
    grouped-GEMM write-up, section 3.3).  Small-integer tokens and weights (over 16) keep every
    sum exact in float64, so both sides round the same values."""
    H, I, n = 64, 48, (7, 9)
    E = len(n)
    rng = np.random.default_rng(5)
    x = rng.integers(-3, 4, (sum(n), H)).astype(np.float64)
    w13 = rng.integers(-4, 5, (E * H, 2 * I)).astype(np.float64) / 16
    w2 = rng.integers(-4, 5, (E * I, H)).astype(np.float64) / 16
    cs = np.concatenate([[0], np.cumsum(n)])
    r = F.grouped_swiglu_ffn(F.f64_to_bf16_bits(x), F.f64_to_bf16_bits(w13), F.f64_to_bf16_bits(w2), cs, H, I)
    t64 = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    bf = lambda t: t.to(torch.bfloat16).to(torch.float64).numpy()
    cast_moved = [False, False]  # each cast changes some value here, so a missing one shows
    for e in range(E):
        s, t = cs[e], cs[e + 1]
        gate, up = (t64(x[s:t]) @ t64(w13[e * H:(e + 1) * H])).split(I, dim=1)
        sw = torch.nn.functional.silu(gate) * up
        assert np.array_equal(r["sw"][s:t], bf(sw))
        down = t64(r["sw"][s:t]) @ t64(w2[e * I:(e + 1) * I])
        assert np.array_equal(r["result"][s:t], bf(down))
        cast_moved[0] |= not np.array_equal(bf(sw), sw.numpy())
        cast_moved[1] |= not np.array_equal(bf(down), down.numpy())
    assert all(cast_moved)


@pytest.mark.parametrize("counts", [(0, 1, 2, 4, 8, 16, 32, 0), (5, 0, 3), (1,)])
def test_against_torch_float64_restatement(counts):
    spec = W.FfnSpec("t", H=128, I=64, E=len(counts), counts=counts, scale=0.3, seed=len(counts))
    inp = W.make_ffn_inputs(spec)
    r = F.grouped_swiglu_ffn(_bits(inp["sorted_tokens"]), _bits(inp["w13_flat"]), _bits(inp["w2_flat"]),
                             inp["expert_cumsum"].numpy(), spec.H, spec.I)
    x = inp["sorted_tokens"].double()
    w13 = inp["w13_flat"].double().view(spec.E, spec.H, 2 * spec.I)
    w2 = inp["w2_flat"].double().view(spec.E, spec.I, spec.H)
    ref = torch.zeros(x.shape[0], spec.H, dtype=torch.float64)
    cs = inp["expert_cumsum"].tolist()
    for e in range(spec.E):
        s, t = cs[e], cs[e + 1]
        gate, up = (x[s:t] @ w13[e]).split(spec.I, dim=1)
        ref[s:t] = (torch.nn.functional.silu(gate) * up) @ w2[e]  # no bf16 steps
    assert np.all(np.abs(r["result"] - ref.numpy()) <= F.tolerance(r["result"], r["absb"]))
    assert np.abs(r["result"] - ref.numpy()).max() > 0  # the bf16 steps are visible


def test_workload_shapes():
    s = W.ffn_config("model")
    assert sum(s.counts) == 4096 and len(s.counts) == 256
    t = W.ffn_config("test")
    assert t.counts == (0, 1, 2, 4, 8, 16, 32, 0)
