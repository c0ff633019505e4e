"""The committed ncu record that bench.py reads its DRAM traffic from
(profiles/gemm_kernel_traffic.json): each workload's entry names the source hash of the
kernel it was captured on, and bench.py reports that traffic only while the current sources
hash the same, so the `roofline.traffic` of a bench line belongs to the kernel it timed
(skipped, not failed, once a kernel change has made an entry stale)."""
import json
import os
import re

import pytest

import bench
from moe_grouped_gemm_mxfp8_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SPECS = {s.name.split()[0]: s for s in [W.config(i) for i in range(1, 6)] +
         [W.large_small_config(), W.mxfp4_config(), W.mxfp4_small_config()]}


def _record():
    if not os.path.exists(bench.PROFILE_RECORD):
        pytest.skip("no profile record committed")
    return json.load(open(bench.PROFILE_RECORD))


def test_record_entries_are_complete():
    rec = _record()
    for name, r in rec["workloads"].items():
        assert name in SPECS, name
        for key in ("source_sha256_16", "traffic_bytes_per_launch", "summary", "commands"):
            assert key in r, (name, key)
        assert os.path.exists(os.path.join(ROOT, "profiles", r["summary"])), r["summary"]
        assert all(re.match(r"(python bench\.py|ncu )", c) for c in r["commands"]), name
        assert all("_work" not in c for c in r["commands"]), name


@pytest.mark.parametrize("name", sorted(SPECS))
def test_committed_traffic_belongs_to_the_current_kernel(name):
    rec = _record()
    if name not in rec["workloads"]:
        pytest.skip(f"{name}: no capture")
    traffic = bench._profiled_traffic(SPECS[name].name)
    if traffic is None:  # bench.py then reports null; a new capture brings the figure back
        pytest.skip(f"{name}: the record predates the current kernel sources")
    # DRAM bytes at or a little above the algorithmic bytes of the workload
    assert 1.0 <= traffic / W.algorithmic_bytes(SPECS[name]) < 1.1


def test_traffic_is_withheld_for_runs_set_up_otherwise():
    for s in SPECS.values():
        assert bench._profiled_traffic(s.name, as_captured=False) is None
    assert bench._profiled_traffic("C9 no such workload") is None


def test_summaries_give_their_command():
    for fn in os.listdir(os.path.join(ROOT, "profiles")):
        if not fn.endswith(".md"):
            continue
        text = open(os.path.join(ROOT, "profiles", fn)).read()
        assert re.search(r"^\s+(python bench\.py|ncu )", text, re.M), fn
        assert "_work" not in text, fn
