"""CPU oracle for the grouped SwiGLU expert FFN (llada2_moe_grouped_gemm).

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).

What it computes (LLaDA2.0-mini grouped-GEMM write-up, section 3.1 input layout
and section 3.2-3.3 per-expert flow):

    expert e owns sorted_tokens rows [cumsum[e], cumsum[e+1])
    gate_up = x_e @ w13_e,   w13_e = w13_flat[e*H:(e+1)*H, :]     ([n_e, 2I])
    gate = gate_up[:, :I],  up = gate_up[:, I:]
    sw   = bf16( SiLU(gate) * up ),  SiLU(g) = g / (1 + exp(-g))
    down = sw @ w2_e,        w2_e = w2_flat[e*I:(e+1)*I, :]        ([n_e, H])
    result rows = bf16(down)

The page accumulates in FP32 and casts sw and the result to BF16; here every
product and sum is done in float64 and only those two casts (round to nearest,
ties to even) are applied, so the oracle is the exact value of the page's
formula up to those two prescribed roundings.  Rows outside every expert range
are left as they are in `result_init`.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> nearest bfloat16 value (ties to even), returned as float64.
    bfloat16 keeps 8 significant bits; values here are far from its range limits."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m * 2^e, 0.5 <= |m| < 1
    r = np.round(m * 256.0)               # numpy rounds half to even
    return np.ldexp(r / 256.0, e)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    r = round_bf16(x).astype(np.float32)  # exact: r has at most 8 significant bits
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def grouped_swiglu_ffn(sorted_tokens, w13_flat, w2_flat, expert_cumsum, H: int, I: int, result_init=None):
    """All arrays are bfloat16 bit patterns (uint16) except expert_cumsum.
    Returns dict(result=float64 [N, H] (bf16 values), absb=float64 [N, H], sw=float64 [N, I]).
    absb[t, h] = sum_i |sw[t, i]| * |w2_e[i, h]| bounds how far an error in sw can move a result."""
    x = bf16_to_f64(sorted_tokens)
    w13 = bf16_to_f64(w13_flat)
    w2 = bf16_to_f64(w2_flat)
    cs = np.asarray(expert_cumsum, dtype=np.int64)
    E = cs.size - 1
    N = x.shape[0]
    res = np.zeros((N, H)) if result_init is None else bf16_to_f64(result_init).copy()
    absb = np.zeros((N, H))
    sw_all = np.zeros((N, I))
    for e in range(E):
        s, t = int(cs[e]), int(cs[e + 1])
        if t <= s:
            continue
        gu = x[s:t] @ w13[e * H:(e + 1) * H]
        sw = round_bf16(silu(gu[:, :I]) * gu[:, I:])
        w2e = w2[e * I:(e + 1) * I]
        res[s:t] = round_bf16(sw @ w2e)
        absb[s:t] = np.abs(sw) @ np.abs(w2e)
        sw_all[s:t] = sw
    return dict(result=res, absb=absb, sw=sw_all)


def tolerance(result: np.ndarray, absb: np.ndarray) -> np.ndarray:
    """Bound on |gpu - oracle| per result element: one bf16 step of the result
    (2^-7 relative: two values a rounding apart land on adjacent bf16 values), one
    bf16 step of every sw that feeds it (2^-7 * absb, with 10% margin for FP32
    accumulation), and 1e-7 absolute."""
    return 2.0 ** -7 * np.abs(result) + 1.1 * 2.0 ** -7 * absb + 1e-7
