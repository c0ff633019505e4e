"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one part of the oracle to an independent source: torch's own
FP8 / E8M0 / bf16 conversions, the OCP format anchors, a float64 numpy matmul,
closed forms, a hand-worked example, or an invariant of the operator
(grouped_matmul_finalize_routing MXFP8 write-up, sections 2.1-2.2, 4.3, 6.3).
"""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_mxfp8_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- decoders
def _torch_decode(codes: np.ndarray, dt) -> np.ndarray:
    t = torch.from_numpy(codes.astype(np.uint8)).view(dt)
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("fmt,dt", [(W.E4M3, torch.float8_e4m3fn), (W.E5M2, torch.float8_e5m2)])
def test_fp8_decode_all_codes_match_torch(fmt, dt):
    codes = np.arange(256)
    ref = _torch_decode(codes, dt)
    got = np.array([oracle.decode_fp8(fmt, int(c)) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def test_e8m0_decode_all_codes_match_torch():
    codes = np.arange(256)
    ref = _torch_decode(codes, torch.float8_e8m0fnu)
    got = np.array([oracle.decode_e8m0(int(c)) for c in codes])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(ref[:255], got[:255])


def test_format_anchor_values():
    # OCP 8-bit FP / MX specification anchors
    assert oracle.decode_fp8(W.E4M3, 0x7E) == 448.0          # E4M3 max normal
    assert oracle.decode_fp8(W.E4M3, 0x01) == 2.0 ** -9      # E4M3 min subnormal
    assert oracle.decode_fp8(W.E4M3, 0x08) == 2.0 ** -6      # E4M3 min normal
    assert math.isnan(oracle.decode_fp8(W.E4M3, 0x7F))       # S.1111.111 is NaN
    assert oracle.decode_fp8(W.E4M3, 0xB8) == -1.0
    assert oracle.decode_fp8(W.E5M2, 0x7B) == 57344.0        # E5M2 max normal
    assert oracle.decode_fp8(W.E5M2, 0x01) == 2.0 ** -16     # E5M2 min subnormal
    assert oracle.decode_fp8(W.E5M2, 0x7C) == math.inf
    assert oracle.decode_fp8(W.E5M2, 0xFC) == -math.inf
    assert math.isnan(oracle.decode_fp8(W.E5M2, 0x7D))
    assert oracle.decode_e8m0(127) == 1.0
    assert oracle.decode_e8m0(0) == 2.0 ** -127
    assert oracle.decode_e8m0(254) == 2.0 ** 127
    assert math.isnan(oracle.decode_e8m0(255))


def test_bf16_decode_matches_torch():
    bits = np.random.default_rng(0).integers(0, 1 << 16, 4096).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite only
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode_bf16(int(b)) for b in bits])
    assert np.array_equal(ref, got)


# OCP Microscaling Formats (MX) v1.0, FP4 E2M1 element table: codes 0..7 are
# 0, 0.5, 1, 1.5, 2, 3, 4, 6; codes 8..15 the same magnitudes negated.
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_decode_matches_ocp_table():
    got = [oracle.decode_fp8(W.E2M1, c) for c in range(16)]
    assert got == E2M1_VALUES
    assert [math.copysign(1.0, v) for v in got[8:]] == [-1.0] * 8  # the sign bit of -0 too
    # only the low nibble is a code: higher bits of the byte are ignored
    assert [oracle.decode_fp8(W.E2M1, 0xF0 | c) for c in range(16)] == E2M1_VALUES


def test_every_e2m1_value_is_an_e4m3_value():
    """Each FP4 value is exactly representable in E4M3, so an FP4 problem equals
    the same problem with its codes widened to E4M3 bytes."""
    vals = torch.tensor(E2M1_VALUES, dtype=torch.float64)
    assert torch.equal(vals.to(torch.float8_e4m3fn).to(torch.float64), vals)


# ----------------------------------------------------------------------------- helpers
def _spec(**kw) -> W.Spec:
    base = dict(name="tiny", batch=4, M=12, K=128, N=24, E=3, seed=7)
    base.update(kw)
    return W.Spec(**base)


def _run(spec, inp):
    return oracle.run(oracle.problem_from_spec(spec, inp))


def _torch_golden(spec: W.Spec, inp) -> np.ndarray:
    """Independent restatement of the write-up's golden (section 6.3) with torch
    float64 ops: decode through torch's float8 dtypes, expand the E8M0 scales by
    32 along K, one matmul per expert, multiply by logit, index_add_ into out,
    then add the weighted shared input."""
    M, K, N, E = spec.M, spec.K, spec.N, spec.E
    f8 = {W.E4M3: torch.float8_e4m3fn, W.E5M2: torch.float8_e5m2}

    def decode(t, fmt):
        if fmt != W.E2M1:
            return t.view(f8[fmt]).to(torch.float64)
        # unpack the nibbles (even element low) and look them up in the OCP FP4 table
        codes = torch.stack([t & 15, t >> 4], dim=-1).reshape(*t.shape[:-1], -1).long()
        return torch.tensor(E2M1_VALUES, dtype=torch.float64)[codes]

    x1 = decode(inp["x1"], spec.x1_dtype)
    x2 = decode(inp["x2"], spec.x2_dtype)
    if spec.transpose_x2:
        x2 = x2.transpose(1, 2)  # -> [E, K, N]
    e8 = lambda b: b.view(torch.float8_e8m0fnu).to(torch.float64)
    sx = e8(inp["pertoken_scale"]).reshape(M, -1).repeat_interleave(32, dim=1)[:, :K]
    sc = e8(inp["scale"])
    if not spec.scale_per_expert:
        sc = sc.unsqueeze(0).expand(E, *sc.shape)
    if spec.transpose_x2:  # [E, N, Ks, 2] -> [E, N, 2Ks] -> [E, K, N]
        sw = sc.reshape(E, N, -1).repeat_interleave(32, dim=2)[:, :, :K].transpose(1, 2)
    else:  # [E, Ks, N, 2] -> [E, 2Ks, N]
        sw = sc.permute(0, 1, 3, 2).reshape(E, -1, N).repeat_interleave(32, dim=1)[:, :K, :]
    a = x1 * sx
    b = x2 * sw
    out = inp["out"].to(torch.float64).clone()
    counts = inp["group_list"].clone()
    if spec.group_list_type == 0:
        counts = torch.diff(counts, prepend=torch.zeros(1, dtype=counts.dtype))
    start = 0
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        mm = a[start:start + c] @ b[e]
        if inp.get("bias") is not None:  # bias reading: added per expert and column before the logit
            mm = mm + inp["bias"][e].to(torch.float64)[None, :]
        if inp["logit"] is not None:
            mm = mm * inp["logit"][start:start + c].to(torch.float64)[:, None]
        out.index_add_(0, inp["row_index"][start:start + c], mm)
        start += c
    if inp["shared_input"] is not None:
        R = inp["shared_input"].shape[0]
        out[spec.shared_offset:spec.shared_offset + R] += spec.shared_weight * inp["shared_input"].to(torch.float64)
    return out.numpy()


# ----------------------------------------------------------------------------- contraction pins
def test_textbook_gemm_special_case():
    """Unit scales, one expert holding every token, logit 1, identity rows and no
    shared input reduce the operator to out = A @ B (float64 numpy matmul of
    torch-decoded values)."""
    spec = _spec(batch=12, M=12, K=192, N=40, E=1, scale_lo=127, scale_hi=127, logit="none",
                 shared_rows=0, rows="mod")
    inp = W.make_inputs(spec)
    out, absb, flags = _run(spec, inp)
    A = inp["x1"].view(torch.float8_e4m3fn).to(torch.float64).numpy()
    B = inp["x2"].view(torch.float8_e4m3fn).to(torch.float64).numpy()[0]
    ref = A @ B
    assert flags == 0
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(absb, np.abs(A) @ np.abs(B), rtol=1e-13, atol=1e-12)


def test_small_integer_values_are_exact():
    """FP8 codes of small integers with power-of-two scales give exact integer
    results; compared with an integer matmul."""
    rng = np.random.default_rng(3)
    M, K, N = 8, 96, 16
    ints = np.array([-4, -3, -2, -1, 0, 1, 2, 3, 4])
    to_code = {v: int(torch.tensor([float(v)]).to(torch.float8_e4m3fn).view(torch.uint8)) for v in ints}
    A = rng.choice(ints, size=(M, K))
    B = rng.choice(ints, size=(K, N))
    spec = _spec(batch=M, M=M, K=K, N=N, E=1, logit="none", shared_rows=0)
    inp = W.make_inputs(spec)
    inp["x1"] = torch.tensor(np.vectorize(to_code.get)(A), dtype=torch.uint8)
    inp["x2"] = torch.tensor(np.vectorize(to_code.get)(B), dtype=torch.uint8).reshape(1, K, N)
    inp["scale"].fill_(127)
    inp["pertoken_scale"].fill_(128)  # every token value doubled
    out, _, _ = _run(spec, inp)
    assert np.array_equal(out, 2 * (A @ B).astype(np.float64))


@pytest.mark.parametrize("transpose", [False, True])
def test_one_scale_per_32_k_elements(transpose):
    """All-ones FP8 data with distinct scales on each 32-element half of each
    64-element block: the result is 32 * sum over halves of 2^(sx-127)*2^(sw-127)
    (closed form; a 64-element or permuted reading gives another number)."""
    M, K, N = 2, 128, 4
    spec = _spec(batch=M, M=M, K=K, N=N, E=1, logit="none", shared_rows=0, transpose_x2=transpose)
    inp = W.make_inputs(spec)
    inp["x1"].fill_(0x38)  # 1.0
    inp["x2"].fill_(0x38)
    sx = np.array([[127, 128, 129, 126], [125, 127, 130, 127]])  # [token, k/32]
    inp["pertoken_scale"] = torch.tensor(sx.reshape(M, 2, 2), dtype=torch.uint8)
    sw = np.array([[127 + ((n + j) % 3) for j in range(4)] for n in range(N)])  # [n, k/32]
    if transpose:
        inp["scale"] = torch.tensor(sw.reshape(N, 2, 2), dtype=torch.uint8)
    else:
        inp["scale"] = torch.tensor(sw.reshape(N, 2, 2).transpose(1, 0, 2).copy(), dtype=torch.uint8)
    out, _, _ = _run(spec, inp)
    exp = np.array([[32 * sum(2.0 ** (sx[t, j] - 127) * 2.0 ** (sw[n, j] - 127) for j in range(4))
                     for n in range(N)] for t in range(M)])
    assert np.array_equal(out, exp)


def _golden_inputs(g, type_key, transpose):
    M, K, N, E = g["M"], g["K"], g["N"], g["E"]
    x1 = np.zeros((M, K), np.uint8)
    for t, row in enumerate(g["x1_rows"]):
        k = 0
        for i in range(0, len(row), 2):
            x1[t, k:k + row[i + 1]] = int(row[i], 16)
            k += row[i + 1]
    x2 = np.zeros((E, K, N), np.uint8)
    for e in range(E):
        for n in range(N):
            x2[e, :, n] = int(g["x2_kn"][f"expert{e}"][f"col{n}"], 16)
    sc = np.array(g["scale_pairs_per_col"], np.uint8)  # [N, 2] with Ks = 1
    if transpose:
        x2 = x2.transpose(0, 2, 1).copy()
        scale = sc.reshape(N, 1, 2)
    else:
        scale = sc.reshape(1, N, 2)
    shared = np.array([[int(b, 16) for b in r] for r in g["shared_input_bf16_bits"]], np.uint16)
    return oracle.Problem(
        M=M, K=K, N=N, E=E, batch=g["batch"], x1=x1, x2=x2, scale=scale,
        pertoken_scale=np.array(g["pertoken_scale_pairs"], np.uint8).reshape(M, 1, 2),
        group_list=np.array(g[type_key], np.int64), row_index=np.array(g["row_index"], np.int64),
        out=np.array(g["out_init"], np.float32), transpose_x2=transpose,
        group_list_type=1 if type_key == "group_list_type1" else 0,
        logit=np.array(g["logit"], np.float32), shared_input=shared,
        shared_offset=g["shared_input_offset"], shared_weight=g["shared_input_weight"])


@pytest.mark.parametrize("type_key", ["group_list_type1", "group_list_type0"])
@pytest.mark.parametrize("transpose", [False, True])
def test_hand_worked_example(type_key, transpose):
    g = json.load(open(os.path.join(GOLDEN, "worked_example_mxfp8.json")))
    p = _golden_inputs(g, type_key, transpose)
    out, absb, flags = oracle.run(p)
    assert flags == 0
    assert np.array_equal(out, np.array(g["expected_out"]))
    assert np.array_equal(absb, np.array(g["expected_absbound"]))
    # the shared values recorded in the fixture are what the bf16 bits mean
    bits = [[int(b, 16) for b in r] for r in g["shared_input_bf16_bits"]]
    assert [[oracle.decode_bf16(b) for b in r] for r in bits] == g["shared_input_values"]


TINY = [
    dict(),
    dict(transpose_x2=True),
    dict(x1_dtype=W.E5M2, x2_dtype=W.E5M2, group_list_type=0, scale_lo=120, scale_hi=134),
    dict(x1_dtype=W.E5M2, x2_dtype=W.E4M3),
    dict(scale_per_expert=True),
    dict(scale_per_expert=True, transpose_x2=True),
    dict(K=96),                      # ceil(K/64) pads the last pair
    dict(K=160, transpose_x2=True),
    dict(K=32, N=8),
    dict(counts="explicit", explicit_counts=(0, 5, 0), M=9),     # zero-token experts, tokens past the groups
    dict(rows="random", shared_rows=2, shared_offset=1, shared_weight=0.7, out_init="randn"),
    dict(logit="none", shared_rows=0),
    dict(bias=True, rows="random", out_init="randn"),
    dict(bias=True, transpose_x2=True, counts="explicit", explicit_counts=(0, 7, 5), M=14),
    dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1),                       # MXFP4, x2 packed along N
    dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, transpose_x2=True),    # x2 packed along K
    dict(x1_dtype=W.E2M1, x2_dtype=W.E4M3, K=96, rows="random"),
    dict(x1_dtype=W.E5M2, x2_dtype=W.E2M1, transpose_x2=True, scale_per_expert=True, bias=True),
]


@pytest.mark.parametrize("kw", TINY, ids=[str(i) for i in range(len(TINY))])
def test_brute_force_against_torch_golden(kw):
    spec = _spec(**kw)
    inp = W.make_inputs(spec)
    out, _, flags = _run(spec, inp)
    ref = _torch_golden(spec, inp)
    assert flags == 0
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("transpose", [False, True])
def test_e2m1_problem_equals_its_e4m3_widening(transpose):
    """Packed FP4 inputs and the same values widened to one E4M3 byte each give
    bit-identical oracle results (exact values, same summation order).  The
    widening unpacks with numpy along each tensor's last dimension, so a swapped
    nibble order or a packing along the wrong dimension in the oracle fails."""
    spec = _spec(x1_dtype=W.E2M1, x2_dtype=W.E2M1, transpose_x2=transpose, rows="random", out_init="randn")
    inp = W.make_inputs(spec)
    out4, absb4, f4 = _run(spec, inp)

    def widen(t):
        a = t.numpy()
        codes = np.stack([a & 15, a >> 4], axis=-1).reshape(*a.shape[:-1], -1)
        vals = torch.from_numpy(np.array(E2M1_VALUES)[codes])
        return vals.to(torch.float8_e4m3fn).view(torch.uint8)

    spec8 = dataclasses.replace(spec, x1_dtype=W.E4M3, x2_dtype=W.E4M3)
    inp8 = dict(inp, x1=widen(inp["x1"]), x2=widen(inp["x2"]))
    out8, absb8, f8 = _run(spec8, inp8)
    assert f4 == f8 == 0
    assert np.array_equal(out4, out8) and np.array_equal(absb4, absb8)
    # and the FP4 codes do reach every value of the table
    assert set(np.unique(inp["x1"].numpy() & 15)) == set(range(16))


# ----------------------------------------------------------------------------- routing pins
def test_expert_ranges_closed_form():
    spec = _spec(E=4, M=10, counts="explicit", explicit_counts=(3, 0, 4, 2))
    inp = W.make_inputs(spec)
    s, e, f = oracle.expert_ranges(oracle.problem_from_spec(spec, inp))
    assert f == 0 and list(s) == [0, 3, 3, 7] and list(e) == [3, 3, 7, 9]
    spec0 = dataclasses.replace(spec, group_list_type=0)
    inp0 = W.make_inputs(spec0)
    assert inp0["group_list"].tolist() == [3, 3, 7, 9]
    s0, e0, f0 = oracle.expert_ranges(oracle.problem_from_spec(spec0, inp0))
    assert f0 == 0 and list(s0) == list(s) and list(e0) == list(e)


@pytest.mark.parametrize("gtype,gl,exp_start,exp_end", [
    (1, [3, -2, 4, 9], [0, 3, 3, 7], [3, 3, 7, 10]),   # negative count, total > M
    (0, [3, 2, 7, 12], [0, 3, 3, 7], [3, 3, 7, 10]),   # decreasing prefix, last > M
    # one fault at a time: each alone raises the flag
    (1, [3, 0, 4, 9], [0, 3, 3, 7], [3, 3, 7, 10]),    # total > M
    (1, [3, -2, 4, 3], [0, 3, 3, 7], [3, 3, 7, 10]),   # negative count
    (0, [3, 2, 7, 10], [0, 3, 3, 7], [3, 3, 7, 10]),   # decreasing prefix
    (0, [3, 3, 7, 12], [0, 3, 3, 7], [3, 3, 7, 10]),   # last prefix > M
])
def test_invalid_group_list_is_flagged_and_clamped(gtype, gl, exp_start, exp_end):
    spec = _spec(E=4, M=10, group_list_type=gtype)
    inp = W.make_inputs(spec)
    inp["group_list"] = torch.tensor(gl, dtype=torch.int64)
    s, e, f = oracle.expert_ranges(oracle.problem_from_spec(spec, inp))
    assert f == oracle.BAD_GROUP_LIST
    assert list(s) == exp_start and list(e) == exp_end


def test_type0_equals_type1():
    spec = _spec(counts="multinomial", M=20, E=5, rows="random")
    a = _run(spec, W.make_inputs(spec))[0]
    spec0 = dataclasses.replace(spec, group_list_type=0)
    b = _run(spec0, W.make_inputs(spec0))[0]
    assert np.array_equal(a, b)


def test_zero_logit_and_zero_shared_weight_leave_out_unchanged():
    spec = _spec(out_init="randn", shared_weight=0.0, rows="random")
    inp = W.make_inputs(spec)
    inp["logit"].zero_()
    out, _, _ = _run(spec, inp)
    assert np.array_equal(out, inp["out"].numpy().astype(np.float64))


def test_linear_in_logit_and_shared_weight():
    spec = _spec(out_init="randn", rows="random", shared_weight=0.75)
    inp = W.make_inputs(spec)
    base = inp["out"].numpy().astype(np.float64)
    d1 = _run(spec, inp)[0] - base
    inp2 = dict(inp, logit=inp["logit"] * 2)  # powers of two keep every step exact
    d2 = _run(dataclasses.replace(spec, shared_weight=1.5), inp2)[0] - base
    np.testing.assert_allclose(d2, 2 * d1, rtol=1e-12, atol=1e-9)


def test_permuting_tokens_within_an_expert_changes_nothing():
    spec = _spec(counts="explicit", explicit_counts=(5, 4, 3), M=12, rows="mod", batch=12)
    inp = W.make_inputs(spec)
    out = _run(spec, inp)[0]
    perm = torch.cat([torch.randperm(5, generator=torch.Generator().manual_seed(1)),
                      5 + torch.randperm(4, generator=torch.Generator().manual_seed(2)),
                      9 + torch.randperm(3, generator=torch.Generator().manual_seed(3))])
    inp_p = dict(inp, x1=inp["x1"][perm], pertoken_scale=inp["pertoken_scale"][perm],
                 logit=inp["logit"][perm], row_index=inp["row_index"][perm])
    # rows are distinct here, so the addition order within each element is unchanged
    assert np.array_equal(_run(spec, inp_p)[0], out)


def test_tokens_outside_groups_and_bad_rows():
    spec = _spec(counts="explicit", explicit_counts=(2, 0, 3), M=9, rows="mod", batch=9)
    inp = W.make_inputs(spec)
    out, absb, flags = _run(spec, inp)
    assert flags == 0
    init = inp["out"].numpy().astype(np.float64)
    shared = spec.shared_weight * inp["shared_input"].to(torch.float64).numpy()
    # tokens 5..8 lie past the last group: their rows only see init + shared
    assert np.array_equal(out[5:], init[5:] + shared[5:])
    assert np.all(absb[5:] == 0)
    inp["row_index"][1] = 99
    out2, _, flags2 = _run(spec, inp)
    assert flags2 == oracle.BAD_ROW_INDEX
    assert np.array_equal(out2[1], init[1] + shared[1])
    assert np.array_equal(np.delete(out2, 1, 0), np.delete(out, 1, 0))


def test_nan_scale_code_poisons_exactly_its_outputs():
    spec = _spec(E=1, M=4, batch=4, logit="none", shared_rows=0)
    inp = W.make_inputs(spec)
    inp["pertoken_scale"][2, 1, 0] = 255  # token 2, k in [64, 96)
    inp["scale"][0, 5, 1] = 255           # column 5, k in [32, 64)
    out, _, _ = _run(spec, inp)
    nan = np.isnan(out)
    exp = np.zeros_like(nan)
    exp[2, :] = True
    exp[:, 5] = True
    assert np.array_equal(nan, exp)


def test_k_tail_padding_scale_is_ignored():
    """K=96: the second half of the last scale pair covers k in [96,128), past K;
    a NaN code there must not reach the result (padding reading)."""
    spec = _spec(K=96)
    inp = W.make_inputs(spec)
    out, _, _ = _run(spec, inp)
    inp["pertoken_scale"][:, 1, 1] = 255
    inp["scale"][1, :, 1] = 255
    out2, _, _ = _run(spec, inp)
    assert np.array_equal(out, out2)


def test_bias_closed_form():
    """Zero activations leave only the bias: out[r,n] = init + sum over the row's
    tokens of logit * bias[expert, n] (bf16 values chosen exactly representable)."""
    spec = _spec(bias=True, rows="mod", batch=12, shared_rows=0, out_init="randn")
    inp = W.make_inputs(spec)
    inp["x1"].zero_()
    bias = torch.tensor([[0.5 * (e + 1) - 0.25 * (n % 5) for n in range(spec.N)] for e in range(spec.E)])
    inp["bias"] = bias.to(torch.bfloat16)
    out, absb, _ = _run(spec, inp)
    exp = inp["out"].numpy().astype(np.float64).copy()
    counts = inp["group_list"].tolist()
    t = 0
    for e, c in enumerate(counts):
        for _ in range(c):
            exp[int(inp["row_index"][t])] += float(inp["logit"][t]) * bias[e].double().numpy()
            t += 1
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-12)


def test_sampled_equals_full():
    spec = _spec(rows="random", out_init="randn", shared_rows=3, shared_offset=1, shared_weight=0.7, bias=True)
    inp = W.make_inputs(spec)
    p = oracle.problem_from_spec(spec, inp)
    out, absb, _ = oracle.run(p)
    rr, cc = np.meshgrid(np.arange(spec.batch), np.arange(spec.N), indexing="ij")
    v, b, _ = oracle.run_sampled(p, rr.ravel(), cc.ravel())
    assert np.array_equal(v.reshape(out.shape), out)
    assert np.array_equal(b.reshape(out.shape), absb)


def test_benchmark_recipes():
    """The five workload recipes produce the documented shapes and routing."""
    c = [W.expert_counts(W.config(i)) for i in range(1, 6)]
    assert c[0].tolist() == [16] * 8 and c[1].tolist() == [16] * 16 and c[2].tolist() == [24] * 32
    assert int(c[3].sum()) == 768 and int((c[3] == 0).sum()) >= 1 and int(c[3][0]) == int(c[3].max())
    assert int(c[4].sum()) == 4096 and c[4].numel() == 256
    s3 = W.config(3)
    gl = W.group_list_from_counts(c[2], s3.group_list_type)
    assert gl.tolist() == list(range(24, 769, 24))
