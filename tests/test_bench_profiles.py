"""The committed ncu summaries that bench.py reads its DRAM traffic from: each names the
source hash of the kernel it was captured on, and bench.py reports that traffic only while
the current sources hash the same, so the `roofline.traffic` of a bench line belongs to the
kernel it timed (skipped, not failed, once a kernel change has made a summary stale)."""
import os
import re

import pytest

import bench
from moe_grouped_gemm_mxfp8_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("spec", [W.config(2), W.mxfp4_small_config(), W.mxfp4_config()],
                         ids=["C2", "MXFP4-E32", "C5-MXFP4"])
def test_committed_traffic_belongs_to_the_current_kernel(spec):
    traffic = bench._profiled_traffic(spec.name)
    if traffic is None:  # bench.py then reports null; a new capture brings the figure back
        pytest.skip(f"{spec.name}: the summary predates the current kernel sources")
    # DRAM bytes at or a little above the algorithmic bytes of the workload
    assert 1.0 <= traffic / W.algorithmic_bytes(spec) < 1.1


def test_traffic_is_withheld_for_runs_set_up_otherwise():
    assert bench._profiled_traffic(W.config(2).name, as_captured=False) is None
    assert bench._profiled_traffic(W.config(1).name) is None  # no capture of this workload


def test_summaries_give_their_command():
    for fn in os.listdir(os.path.join(ROOT, "profiles")):
        text = open(os.path.join(ROOT, "profiles", fn)).read()
        assert re.search(r"^\s+(python bench\.py|ncu )", text, re.M), fn
        assert "_work" not in text, fn
