"""CPU oracle for the MoE routing step that produces the operator's inputs.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).

What it computes (LLaDA2.0-mini grouped-GEMM write-up, section 5.2: the
flattened expert ids are argsorted, counted with bincount and prefix-summed,
and the tokens gathered in that order; the grouped-matmul-finalize-routing
operator then plays the role of the inverse permutation and of the top-k
weighted sum, write-up on grouped_matmul_finalize_routing, section 2.2):

    flat index f = b * topk + k,  expert id[f] = topk_ids[b, k]
    order: entries sorted by expert id, ties in ascending f (a stable sort);
           entries whose id lies outside [0, E) are dropped from every group and
           placed after all routed entries, in ascending f (reading: invalid ids
           route nowhere; the error flag reports them)
    for output position p holding entry f:
        perm[p] = f, row_index[p] = f // topk, logit[p] = topk_weights[b, k] (1 if absent),
        x1[p, :] = x[f // topk, :], pertoken_scale[p] = x_scale[f // topk]
    group_list = per-expert counts (type 1) or their inclusive prefix sums (type 0)
"""
from __future__ import annotations

import numpy as np

BAD_EXPERT_ID = 1


def moe_route(topk_ids, topk_weights, x, x_scale, E: int, group_list_type: int = 1):
    """Returns dict(perm, x1, pertoken_scale, group_list, row_index, logit, flags)."""
    ids = np.asarray(topk_ids).astype(np.int64)
    batch, topk = ids.shape
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    key = np.where(valid, flat, E)                      # invalid ids sort last
    perm = np.argsort(key, kind="stable").astype(np.int64)
    counts = np.bincount(flat[valid], minlength=E).astype(np.int64)
    group_list = counts if group_list_type == 1 else np.cumsum(counts)
    src_row = perm // topk
    x = np.asarray(x)
    xs = np.asarray(x_scale)
    w = None if topk_weights is None else np.asarray(topk_weights, dtype=np.float32).reshape(-1)
    return dict(
        perm=perm,
        x1=x[src_row],
        pertoken_scale=xs[src_row],
        group_list=group_list.astype(np.int64),
        row_index=src_row.astype(np.int64),
        logit=np.ones(perm.size, np.float32) if w is None else w[perm],
        flags=0 if bool(valid.all()) else BAD_EXPERT_ID,
    )
