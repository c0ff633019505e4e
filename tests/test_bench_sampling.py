"""The CPU baseline's column sample: the oracle on output columns [0, ncols) of a
workload equals those columns of the oracle on the whole workload, for every x2 layout
and element format (packed E2M1 holds two columns per byte when x2 is not transposed)."""
import dataclasses

import numpy as np
import pytest

import bench
import oracle
from moe_grouped_gemm_mxfp8_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


BASE = W.Spec("sample", batch=12, M=24, K=96, N=40, E=3, rows="random", shared_rows=5, shared_offset=2,
              shared_weight=0.5, out_init="randn", seed=31)


@pytest.mark.parametrize("kw", [
    dict(),
    dict(transpose_x2=True),
    dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1),
    dict(x1_dtype=W.E2M1, x2_dtype=W.E2M1, transpose_x2=True),
    dict(x2_dtype=W.E2M1, scale_per_expert=True),
    dict(bias=True, transpose_x2=True),
])
def test_column_sample_equals_full_run(kw):
    spec = dataclasses.replace(BASE, **kw)
    inp = W.make_inputs(spec)
    full, absb, _ = oracle.run(bench._oracle_problem(spec, inp, spec.N))
    ncols = 16
    part, absb_p, _ = oracle.run(bench._oracle_problem(spec, inp, ncols))
    assert np.array_equal(part, full[:, :ncols])
    assert np.array_equal(absb_p, absb[:, :ncols])
