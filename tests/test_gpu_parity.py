"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Tolerance (per element): |gpu - oracle| <= 1e-4 * absb + 1e-6, absb = sum over the
element's tokens of |logit| * sum_k |a_k b_k| (oracle.tolerance: the operator's stated
bound, per token); NaN positions must match exactly; device error bits must equal the
oracle's flags.  Every benchmark workload is compared element by element in full.
"""
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

import _parity_report
import oracle
from moe_grouped_gemm_mxfp8_gb300 import binding as B
from moe_grouped_gemm_mxfp8_gb300 import build as build_mod
from moe_grouped_gemm_mxfp8_gb300 import workloads as W

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    oracle.build()
    B.load()


def _dev(inp, row_i32=False):
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    if row_i32:
        d["row_index"] = d["row_index"].to(torch.int32)
    return d


def gpu_run(spec, inp, deterministic=False, prepared=True, row_i32=False, d=None):
    d = d or _dev(inp, row_i32)
    prob = B.problem_from_spec(spec, deterministic, B.INDEX_I32 if row_i32 else B.INDEX_I64)
    prep = B.prepare_weights(prob, d["x2"], d["scale"]) if prepared else None
    out = d["out"].clone()
    ws = B.run(prob, d, out, prepared=prep)
    bits = B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return out.cpu().numpy().astype(np.float64), bits


def assert_close(got, ref, bound, what=""):
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"NaN mismatch at {np.argwhere(nan_g != nan_r)[:5]}"
    m = ~nan_r
    err = np.abs(got[m] - ref[m])
    ratio = err / bound[m]
    worst = int(np.argmax(ratio)) if ratio.size else 0
    if ratio.size:
        _parity_report.record(ratio.max(), what)
    assert ratio.size == 0 or ratio.max() <= 1.0, (
        f"max err/bound {ratio.max():.3g} (err {err[worst]:.3g}, bound {bound[m][worst]:.3g}, ref {ref[m][worst]:.6g})")


def check_full(spec, inp, **kw):
    got, bits = gpu_run(spec, inp, **kw)
    ref, absb, flags = oracle.run(oracle.problem_from_spec(spec, inp))
    assert_close(got, ref, oracle.tolerance(ref, absb))
    assert bits == flags
    return got, ref


def _spec(**kw):
    base = dict(name="t", batch=16, M=40, K=256, N=320, E=4, seed=11)
    base.update(kw)
    return W.Spec(**base)


# ----------------------------------------------------------------------------- worked example
@pytest.mark.parametrize("transpose", [False, True])
def test_hand_worked_example(transpose):
    g = json.load(open(os.path.join(GOLDEN, "worked_example_mxfp8.json")))
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
    sc = np.array(g["scale_pairs_per_col"], np.uint8)
    if transpose:
        x2, scale = x2.transpose(0, 2, 1).copy(), sc.reshape(N, 1, 2)
    else:
        scale = sc.reshape(1, N, 2)
    shared = torch.tensor(g["shared_input_values"], dtype=torch.float32).to(torch.bfloat16)
    spec = W.Spec("golden", batch=g["batch"], M=M, K=K, N=N, E=E, transpose_x2=transpose,
                  shared_weight=g["shared_input_weight"])
    inp = dict(x1=torch.from_numpy(x1), x2=torch.from_numpy(x2), scale=torch.from_numpy(scale),
               pertoken_scale=torch.tensor(g["pertoken_scale_pairs"], dtype=torch.uint8).reshape(M, 1, 2),
               group_list=torch.tensor(g["group_list_type1"]), logit=torch.tensor(g["logit"]),
               row_index=torch.tensor(g["row_index"]), shared_input=shared,
               out=torch.tensor(g["out_init"], dtype=torch.float32))
    for det in (False, True):
        got, bits = gpu_run(spec, inp, deterministic=det)
        assert bits == 0
        np.testing.assert_allclose(got, np.array(g["expected_out"]), rtol=0, atol=1e-5)


# ----------------------------------------------------------------------------- small full-oracle cases
SMALL = {
    "basic": dict(),
    "transposed": dict(transpose_x2=True),
    "e5m2_prefix": dict(x1_dtype=W.E5M2, x2_dtype=W.E5M2, group_list_type=0, scale_lo=120, scale_hi=134),
    "mixed_formats": dict(x1_dtype=W.E5M2, x2_dtype=W.E4M3, transpose_x2=True),
    "per_expert_scale": dict(scale_per_expert=True),
    "per_expert_scale_t": dict(scale_per_expert=True, transpose_x2=True, x1_dtype=W.E5M2, x2_dtype=W.E5M2),
    "k96": dict(K=96),
    "k160_t": dict(K=160, transpose_x2=True),
    "k32_n8": dict(K=32, N=8),
    "k16_n1": dict(K=16, N=1),
    "ragged_counts": dict(E=8, M=63, counts="explicit", explicit_counts=(0, 1, 2, 4, 8, 16, 32, 0)),
    "tokens_past_groups": dict(E=3, M=50, counts="explicit", explicit_counts=(10, 0, 20)),
    "random_rows_shared": dict(rows="random", shared_rows=6, shared_offset=5, shared_weight=0.7, out_init="randn"),
    "no_logit_no_shared": dict(logit="none", shared_rows=0),
    "straddle": dict(E=9, M=1344, batch=200, N=256, K=128, rows="random",
                     counts="explicit", explicit_counts=(63, 64, 65, 127, 128, 129, 255, 256, 257)),
    "many_experts": dict(E=300, M=900, batch=300, N=128, K=128, counts="multinomial", rows="random"),
    # bias: added once per (token, column) even when a tile's K range is split over CTAs
    "bias_split_k": dict(E=4, M=60, N=320, K=1024, bias=True, rows="random", out_init="randn"),
    "bias_wide": dict(E=3, M=300, batch=64, N=256, K=256, bias=True, counts="explicit",
                      explicit_counts=(150, 0, 150), rows="random", transpose_x2=True),
    # MXFP4 (E2M1 codes two per byte): tokens and weights both E2M1 with K % 32 == 0 stay packed
    # (kind::mxf4, 256 K per tile); other E2M1 operands are expanded exactly to E4M3
    "mxfp4": dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1),
    "mxfp4_t": dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, transpose_x2=True, rows="random"),
    "mxfp4_k352_bias": dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, K=352, N=200, bias=True, rows="random",
                            out_init="randn"),                 # two K tiles, the second 96 of 256 long
    "mxfp4_k96": dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, K=96, N=130, transpose_x2=True,
                      scale_per_expert=True),                  # one partial tile, padding scale block
    "mxfp4_k1024_split": dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, E=4, M=60, N=320, K=1024, bias=True,
                              rows="random", out_init="randn"),  # K tiles of one column tile split over CTAs
    "mxfp4_k48_expanded": dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, K=48, N=64),  # K % 32 != 0: expanded
    "mxfp4_tokens_e5m2_weights": dict(x1_dtype=W.E2M1, x2_dtype=W.E5M2, K=96),
    "e4m3_tokens_mxfp4_weights": dict(x2_dtype=W.E2M1, transpose_x2=True, scale_per_expert=True, bias=True,
                                      N=255),
    "mxfp4_k16_n2": dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, K=16, N=2, M=7, batch=5),  # 56-byte packed x1
    # K % 16 != 0 (the aclnn V3 constraints and the ceil(K/64) scale layout of section 3.1 admit any
    # K): x1 rows are copied to a 16-byte pitch first (E2M1 codes expanded on the way)
    "k40": dict(K=40),
    "k72_t": dict(K=72, transpose_x2=True, rows="random", out_init="randn"),
    "k200": dict(K=200, E=3, M=70, counts="explicit", explicit_counts=(33, 0, 37), bias=True),
    "k200_t_e5m2": dict(K=200, transpose_x2=True, x1_dtype=W.E5M2, x2_dtype=W.E5M2, group_list_type=0,
                        scale_per_expert=True),
    "k1": dict(K=1, N=130),
    "k8_n3": dict(K=8, N=3, M=9, batch=4),
    "k1032_split": dict(K=1032, E=4, M=60, N=320, rows="random", out_init="randn"),  # K blocks split over CTAs
    "mxfp4_k40": dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, K=40, N=64),
    "mxfp4_tokens_k72_t": dict(x1_dtype=W.E2M1, x2_dtype=W.E4M3, K=72, transpose_x2=True),
    "mxfp4_weights_k200_t": dict(x2_dtype=W.E2M1, K=200, transpose_x2=True, N=130),
    "mxfp4_straddle": dict(E=9, M=1344, batch=200, N=256, K=128, rows="random", x1_dtype=W.E2M1,
                           x2_dtype=W.E2M1, counts="explicit",
                           explicit_counts=(63, 64, 65, 127, 128, 129, 255, 256, 257)),
    # many short segments per CTA (2 K blocks per column tile, 27 items per CTA), 256 and 257
    # experts (the decode's chunked scan), empty experts under both group_list encodings next to
    # experts of exactly 32 tokens (one 32-row box)
    "short_segments": dict(E=64, M=512, batch=512, N=4096, K=256, rows="random"),
    "e256_multinomial": dict(E=256, M=2048, batch=512, N=256, K=384, counts="multinomial", rows="random",
                             transpose_x2=True),
    "e257": dict(E=257, M=2056, batch=512, N=256, K=384, rows="random"),
    "empty_prefix": dict(E=7, M=90, batch=40, N=512, K=512, group_list_type=0, rows="random",
                         counts="explicit", explicit_counts=(0, 32, 5, 0, 17, 1, 32), out_init="randn"),
    "empty_counts": dict(E=7, M=90, batch=40, N=512, K=512, rows="random", shared_rows=8, shared_offset=3,
                         counts="explicit", explicit_counts=(32, 0, 0, 25, 1, 32, 0)),
    # the expert limit (1024: the decode's scans carry over five chunks of its threads), with
    # empty experts, under both group_list encodings, and with Zipf-sized groups (token groups of
    # 128 and the cost-weighted split over 1024 experts)
    "e1024": dict(E=1024, M=3000, batch=1000, N=256, K=256, counts="multinomial", rows="random"),
    "e1024_zipf_prefix": dict(E=1024, M=4000, batch=1000, N=192, K=384, counts="zipf", group_list_type=0,
                              rows="random", out_init="randn"),
    # many routed tokens (40000: 300-odd token groups of up to 128 in a few large experts)
    "many_tokens": dict(E=16, M=40000, batch=8192, N=256, K=256, counts="zipf", zipf_s=0.8, rows="random",
                        shared_rows=64, shared_offset=100),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_atomic(name):
    check_full(_spec(**SMALL[name]), W.make_inputs(_spec(**SMALL[name])))


# k16_n1, mxfp4_k96 (N 130) and e4m3_tokens_mxfp4_weights (N 255): N % 4 != 0, the combine's
# scalar path
@pytest.mark.parametrize("name", ["basic", "transposed", "ragged_counts", "random_rows_shared", "straddle", "k96",
                                  "bias_split_k", "mxfp4_t", "mxfp4_k352_bias", "k16_n1", "mxfp4_k96",
                                  "e4m3_tokens_mxfp4_weights", "k72_t", "k1032_split", "mxfp4_k40", "e1024",
                                  "e1024_zipf_prefix", "many_tokens"])
def test_small_deterministic(name):
    spec = _spec(**SMALL[name])
    inp = W.make_inputs(spec)
    got, _ = check_full(spec, inp, deterministic=True)
    again, _ = gpu_run(spec, inp, deterministic=True)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("tmax", ["32", "64", "128"])
@pytest.mark.parametrize("case", ["straddle", "mxfp4_straddle"])
def test_token_group_widths(tmax, case, monkeypatch):
    monkeypatch.setenv("GMMFR_TMAX", tmax)
    spec = _spec(**SMALL[case])
    check_full(spec, W.make_inputs(spec))


@pytest.mark.parametrize("tmax", ["32", "128"])
@pytest.mark.parametrize("case", ["straddle", "mxfp4_straddle"])
def test_token_group_widths_deterministic(tmax, case, monkeypatch):
    """Deterministic mode with the group width forced: 32 puts experts of up to 257 tokens into
    many 32-token groups (walked group-major, sibling groups far apart), 128 into few; both match
    the oracle and repeat their bits."""
    monkeypatch.setenv("GMMFR_TMAX", tmax)
    spec = _spec(**SMALL[case])
    inp = W.make_inputs(spec)
    got, _ = check_full(spec, inp, deterministic=True)
    again, _ = gpu_run(spec, inp, deterministic=True)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("grid", ["1", "37", "300"])
@pytest.mark.parametrize("case", ["short_segments", "empty_prefix"])
def test_atomic_grids(grid, case, monkeypatch):
    """Atomic mode for any CTA count: one CTA holding every item (the ring wrapping many
    times), CTAs holding ragged item counts, and more CTAs than SMs (two waves)."""
    monkeypatch.setenv("GMMFR_GRID", grid)
    spec = _spec(**SMALL[case])
    check_full(spec, W.make_inputs(spec))


@pytest.mark.parametrize("hint", [8, 50, 200])
def test_expected_tokens_hint(hint):
    """The tiling hint changes the token group width, never the result."""
    spec = _spec(**SMALL["straddle"])
    inp = W.make_inputs(spec)
    d = _dev(inp)
    prob = B.problem_from_spec(spec)
    prob.expected_tokens_per_expert = hint
    prep = B.prepare_weights(prob, d["x2"], d["scale"])
    out = d["out"].clone()
    ws = B.run(prob, d, out, prepared=prep)
    bits = B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    ref, absb, flags = oracle.run(oracle.problem_from_spec(spec, inp))
    assert_close(out.cpu().numpy().astype(np.float64), ref, oracle.tolerance(ref, absb))
    assert bits == flags


def test_int32_row_index_and_raw_weights():
    spec = _spec(rows="random", shared_rows=4, shared_offset=2)
    inp = W.make_inputs(spec)
    check_full(spec, inp, row_i32=True)
    check_full(spec, inp, prepared=False)


def test_m_zero_adds_only_shared():
    spec = _spec(M=0, E=3, counts="explicit", explicit_counts=(0, 0, 0), out_init="randn")
    check_full(spec, W.make_inputs(spec))
    # deterministic mode: an empty row CSR, the combine adds the shared rows alone
    check_full(spec, W.make_inputs(spec), deterministic=True)


def test_nan_scale_code_propagates():
    spec = _spec(E=1, M=8, batch=8, logit="none", shared_rows=0)
    inp = W.make_inputs(spec)
    inp["pertoken_scale"][2, 1, 0] = 255
    inp["scale"][0, 5, 1] = 255
    got, ref = check_full(spec, inp)
    assert np.isnan(got[2]).all() and np.isnan(got[:, 5]).all()


def test_invalid_group_list_sets_error_and_clamps():
    spec = _spec(E=4, M=40, counts="explicit", explicit_counts=(10, 10, 10, 10))
    inp = W.make_inputs(spec)
    inp["group_list"] = torch.tensor([12, -3, 25, 9], dtype=torch.int64)  # negative count, total > M
    got, _ = check_full(spec, inp)
    spec0 = dataclasses.replace(spec, group_list_type=0)
    inp0 = dict(inp, group_list=torch.tensor([12, 8, 30, 45], dtype=torch.int64))  # decreasing, > M
    check_full(spec0, inp0)


def test_bad_row_index_sets_error_and_is_skipped():
    spec = _spec(rows="random")
    inp = W.make_inputs(spec)
    inp["row_index"][3] = spec.batch
    inp["row_index"][7] = -1
    check_full(spec, inp)
    check_full(spec, inp, deterministic=True)


def test_prepared_layout_round_trip():
    """The prepared tiles hold x2 and its scales at the documented positions
    (bit-exact byte work), for both x2 layouts."""
    for transpose in (False, True):
        spec = _spec(K=200 - 200 % 16, N=200, E=2, transpose_x2=transpose)
        inp = W.make_inputs(spec)
        prob = B.problem_from_spec(spec)
        d = _dev(inp)
        buf = B.prepare_weights(prob, d["x2"], d["scale"]).cpu().numpy()
        E, K, N = spec.E, spec.K, spec.N
        NT, KB, Ks = -(-N // 128), -(-K // 128), spec.Ks
        tiles = buf[:E * NT * KB * 16896].reshape(E, NT, KB, 16896)
        x2 = inp["x2"].numpy()
        x2_kn = x2.transpose(0, 2, 1) if transpose else x2  # -> [E, K, N]
        sc = inp["scale"].numpy()
        for e in range(E):
            for j in range(NT):
                for kb in range(KB):
                    t = tiles[e, j, kb]
                    r = np.arange(128)[:, None]
                    c = np.arange(128)[None, :]
                    w = t[(r * 128 + (((c // 16) ^ (r % 8)) * 16) + c % 16)]
                    n, k = j * 128 + r, kb * 128 + c
                    exp = np.where((n < N) & (k < K), x2_kn[e, np.minimum(k, K - 1), np.minimum(n, N - 1)], 0)
                    assert np.array_equal(w, exp)
                    q = np.arange(4)[None, :]
                    s = t[16384 + 16 * (r % 32) + 4 * (r // 32) + q]
                    g = kb * 4 + q
                    nn = np.minimum(j * 128 + r, N - 1)
                    kp, h = np.minimum(g // 2, Ks - 1), g % 2
                    sv = sc[kp, nn, h] if not transpose else sc[nn, kp, h]
                    exp_s = np.where(((j * 128 + r) < N) & (g * 32 < K), sv, 127)
                    assert np.array_equal(s, exp_s)


def test_prepared_e2m1_equals_prepared_e4m3_widening():
    """E2M1 weights paired with FP8 tokens are prepared as the E4M3 tiles of the same
    values: the prepared buffer of packed FP4 x2 is byte-identical to that of x2 widened
    to one E4M3 byte per element (the widening done here with torch's float8 cast)."""
    table = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
    for transpose in (False, True):
        spec = _spec(K=208, N=200, E=2, transpose_x2=transpose, x1_dtype=W.E4M3, x2_dtype=W.E2M1)
        inp = W.make_inputs(spec)
        x2 = inp["x2"]
        codes = torch.stack([x2 & 15, x2 >> 4], dim=-1).reshape(*x2.shape[:-1], -1).long()
        wide = table[codes].to(torch.float8_e4m3fn).view(torch.uint8)
        prob4 = B.problem_from_spec(spec)
        prob8 = B.problem_from_spec(dataclasses.replace(spec, x1_dtype=W.E4M3, x2_dtype=W.E4M3))
        sc = inp["scale"].cuda()
        p4 = B.prepare_weights(prob4, x2.cuda(), sc).cpu()
        p8 = B.prepare_weights(prob8, wide.cuda(), sc).cpu()
        assert p4.numel() == p8.numel() and torch.equal(p4, p8)


def test_prepared_packed_e2m1_layout_round_trip():
    """E2M1 tokens and weights: the prepared tiles keep the codes packed, K pairs per byte
    (element k = 256 kb + 2c in the low nibble of byte c, k + 1 in the high nibble),
    swizzled as the FP8 tiles, then eight scales per row in two 512-byte chunks
    (bit-exact byte work), for both x2 layouts."""
    for transpose in (False, True):
        spec = _spec(K=352, N=200, E=2, transpose_x2=transpose, x1_dtype=W.E2M1, x2_dtype=W.E2M1)
        inp = W.make_inputs(spec)
        prob = B.problem_from_spec(spec)
        buf = B.prepare_weights(prob, inp["x2"].cuda(), inp["scale"].cuda()).cpu().numpy()
        E, K, N = spec.E, spec.K, spec.N
        NT, KB, Ks = -(-N // 128), -(-K // 256), spec.Ks
        assert buf.size >= E * NT * KB * 17408
        tiles = buf[:E * NT * KB * 17408].reshape(E, NT, KB, 17408)
        x2 = inp["x2"].numpy().astype(np.int64)
        # codes as [E, K, N]
        if transpose:  # [E, N, K/2], packed along K
            codes = np.stack([x2 & 15, x2 >> 4], axis=-1).reshape(E, N, K).transpose(0, 2, 1)
        else:          # [E, K, N/2], packed along N
            codes = np.stack([x2 & 15, x2 >> 4], axis=-1).reshape(E, K, N)
        sc = inp["scale"].numpy()
        r = np.arange(128)[:, None]
        c = np.arange(128)[None, :]
        for e in range(E):
            for j in range(NT):
                for kb in range(KB):
                    t = tiles[e, j, kb]
                    byte = t[(r * 128 + (((c // 16) ^ (r % 8)) * 16) + c % 16)].astype(np.int64)
                    n, k = j * 128 + r, kb * 256 + 2 * c
                    ok = (n < N) & (k < K)
                    nn, kk = np.minimum(n, N - 1), np.minimum(k, K - 2)
                    assert np.array_equal(byte & 15, np.where(ok, codes[e, kk, nn], 0))
                    assert np.array_equal(byte >> 4, np.where(ok, codes[e, kk + 1, nn], 0))
                    q = np.arange(8)[None, :]
                    s = t[16384 + 512 * (q // 4) + 16 * (r % 32) + 4 * (r // 32) + q % 4]
                    g = kb * 8 + q
                    kp, h = np.minimum(g // 2, Ks - 1), g % 2
                    sv = sc[kp, nn, h] if not transpose else sc[nn, kp, h]
                    assert np.array_equal(s, np.where((n < N) & (g * 32 < K), sv, 127))


@pytest.mark.parametrize("offset", [1, 4])
def test_unaligned_pertoken_scale(offset):
    """pertoken_scale at a base that is not 4-byte aligned (offset 1: the packer assembles each
    scale word from bytes) or only 4-byte aligned (offset 4: whole-word loads)."""
    spec = _spec(K=1024, N=256, M=40, E=4, rows="random")
    inp = W.make_inputs(spec)
    d = _dev(inp)
    ps = d["pertoken_scale"]
    buf = torch.zeros(ps.numel() + 32, dtype=torch.uint8, device="cuda")
    view = buf[offset:offset + ps.numel()].view(ps.shape)
    view.copy_(ps)
    d["pertoken_scale"] = view
    got, bits = gpu_run(spec, inp, d=d)
    ref, absb, flags = oracle.run(oracle.problem_from_spec(spec, inp))
    assert_close(got, ref, oracle.tolerance(ref, absb))
    assert bits == flags


def test_timeout_path_reports_and_recovers(monkeypatch):
    """A wait that nothing completes gives up after its limit, reports
    GMMFR_DEV_TIMEOUT, and leaves the context usable."""
    spec = _spec()
    inp = W.make_inputs(spec)
    monkeypatch.setenv("GMMFR_TEST_STALL_NS", "20000000")
    _, bits = gpu_run(spec, inp)
    assert bits & B.DEV_TIMEOUT
    monkeypatch.delenv("GMMFR_TEST_STALL_NS")
    check_full(spec, inp)


# ----------------------------------------------------------------------------- benchmark workloads
def _large_inputs(spec):
    """Inputs of a benchmark workload (weights drawn on the device by the same seeded CUDA
    generator as the benchmark's), the device copies, and prepared weights; x2 stays on the
    host only, for the oracle."""
    inp = W.make_inputs(spec, weights_device="cuda")
    d = _dev(inp)
    prep = B.prepare_weights(B.problem_from_spec(spec), d["x2"], d["scale"])
    inp["x2"] = inp["x2"].cpu()
    del d["x2"]
    torch.cuda.empty_cache()
    return inp, d, prep


def _call(spec, d, prep, deterministic=False):
    prob = B.problem_from_spec(spec, deterministic)
    out = d["out"].clone()
    ws = B.run(prob, d, out, prepared=prep)
    bits = B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return out.cpu().numpy().astype(np.float64), bits


@pytest.mark.parametrize("i", [1, 2, 3, 4, 5])
def test_config_full(i):
    """Every output element of benchmark workload i (MXFP8 write-up section 2.1 formula, the
    golden's order of section 6.3), in atomic mode, and for workloads 2, 4 and 5 in
    deterministic mode too (twice: bit-identical)."""
    spec = W.config(i)
    inp, d, prep = _large_inputs(spec)
    ref, absb, flags = oracle.run(oracle.problem_from_spec(spec, inp))
    bound = oracle.tolerance(ref, absb)
    got, bits = _call(spec, d, prep)
    assert_close(got, ref, bound, "atomic")
    assert bits == flags
    if i in (2, 4, 5):
        det, bits = _call(spec, d, prep, deterministic=True)
        assert_close(det, ref, bound, "deterministic")
        assert bits == flags
        again, _ = _call(spec, d, prep, deterministic=True)
        assert np.array_equal(det, again)


def test_mxfp4_large_full():
    """The MXFP4 (packed E2M1) operator at the large shape, every output element."""
    spec = W.mxfp4_config()
    inp, d, prep = _large_inputs(spec)
    got, bits = _call(spec, d, prep)
    ref, absb, flags = oracle.run(oracle.problem_from_spec(spec, inp))
    assert_close(got, ref, oracle.tolerance(ref, absb))
    assert bits == flags


def _schedules():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return [dict(GMMFR_GRID=str(g)) for g in (1, 37, sms)] + \
           [dict(GMMFR_GRID=str(g), GMMFR_REVERSE_UNITS="1") for g in (37, sms)]


# config4, straddle, k200 and mxfp4_straddle hold token groups of 64 or 128, the others groups of
# at most 32
@pytest.mark.parametrize("case", ["config4", "straddle", "k200", "mxfp4_straddle", "bias_split_k", "mxfp4_t",
                                  "ragged_counts"])
def test_deterministic_bits_do_not_depend_on_the_schedule(case, monkeypatch):
    """Deterministic mode (aclnn V3, 确定性计算) gives the same bits whatever the number of
    CTAs (1, 37, one per SM) and whichever order each CTA takes its units in."""
    if case == "config4":
        spec = W.config(4)
        inp, d, prep = _large_inputs(spec)
    else:
        spec = _spec(**SMALL[case])
        inp = W.make_inputs(spec)
        d = _dev(inp)
        prep = B.prepare_weights(B.problem_from_spec(spec), d["x2"], d["scale"])
    base, bits0 = _call(spec, d, prep, deterministic=True)
    for env in _schedules():
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        got, bits = _call(spec, d, prep, deterministic=True)
        for k in env:
            monkeypatch.delenv(k)
        assert bits == bits0
        assert np.array_equal(got, base), f"{env}: {np.count_nonzero(got != base)} elements differ"
    ref, absb, flags = oracle.run(oracle.problem_from_spec(spec, inp))
    assert_close(base, ref, oracle.tolerance(ref, absb))
    assert bits0 == flags


def test_mxfp4_raw_weights_in_call():
    """E2M1 weights prepared inside the call (no prepared buffer)."""
    spec = _spec(**SMALL["mxfp4_t"])
    inp = W.make_inputs(spec)
    got, bits = gpu_run(spec, inp, prepared=False)
    ref, absb, flags = oracle.run(oracle.problem_from_spec(spec, inp))
    assert_close(got, ref, oracle.tolerance(ref, absb))
    assert bits == flags


def test_deterministic_many_tokens():
    """Deterministic mode with 9000 routed tokens over 3000 rows (row CSR of many tokens)."""
    spec = W.Spec("det many tokens", batch=3000, M=9000, K=128, N=256, E=8, rows="random", counts="multinomial",
                  shared_rows=100, shared_offset=7, shared_weight=0.3, out_init="randn", seed=77)
    check_full(spec, W.make_inputs(spec), deterministic=True)


def test_deterministic_rows_of_more_than_2048_tokens():
    """Two output rows holding about 2200 routed tokens each: the combine orders a row's tokens by
    a block-wide minimum per token instead of in shared memory (rows of up to 2048 tokens)."""
    spec = W.Spec("det long rows", batch=2, M=4400, K=64, N=192, E=3, rows="random", counts="multinomial",
                  shared_rows=1, shared_offset=1, shared_weight=0.5, out_init="randn", seed=78)
    inp = W.make_inputs(spec)
    assert np.bincount(inp["row_index"].numpy(), minlength=2).min() > 2048
    got, _ = check_full(spec, inp, deterministic=True)
    again, _ = gpu_run(spec, inp, deterministic=True)
    assert np.array_equal(got, again)


def test_deterministic_unaligned_out_and_shared():
    """out 4 bytes and shared_input 2 bytes past an aligned base (N % 4 == 0): the combine's scalar
    path, with the same results as the vector path bit for bit."""
    spec = _spec(rows="random", shared_rows=6, shared_offset=5, shared_weight=0.7, out_init="randn")
    inp = W.make_inputs(spec)
    d = _dev(inp)
    aligned, _ = check_full(spec, inp, deterministic=True)
    prob = B.problem_from_spec(spec, True)
    prep = B.prepare_weights(prob, d["x2"], d["scale"])
    n_out, n_sh = d["out"].numel(), d["shared_input"].numel()
    out = torch.empty(n_out + 4, device="cuda")[1:1 + n_out].view(d["out"].shape)
    out.copy_(d["out"])
    shared = torch.empty(n_sh + 8, dtype=torch.bfloat16, device="cuda")[1:1 + n_sh].view(d["shared_input"].shape)
    shared.copy_(d["shared_input"])
    ws = B.run(prob, dict(d, shared_input=shared), out, prepared=prep)
    assert B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    assert np.array_equal(out.cpu().numpy().astype(np.float64), aligned)
