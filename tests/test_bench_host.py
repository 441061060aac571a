"""Host-side rules of the benchmark line (no GPU): the roofline's DRAM traffic is reported only while the
kernel sources match those the committed counters were taken on, and the algorithmic work follows the
stated formulas."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("kind,workload", [("maxsim", "joint"), ("maxsim", "maxsim3"), ("pooled", "pooled4")])
def test_committed_traffic_is_reported_while_the_sources_match(kind, workload, monkeypatch):
    record, files = bench.TRAFFIC_RECORDS[kind]
    with open(os.path.join(ROOT, "profiles", record)) as f:
        d = json.load(f)
    assert len(d["source_hash"]) == 16 and all(n.endswith((".cu", ".cuh")) for n in files)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda files=None: d["source_hash"])
    assert bench.committed_traffic(workload, kind) == d["per_launch_bytes"][workload] > 0


def test_traffic_is_null_once_a_kernel_source_changes(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_hash", lambda files=None: "0000000000000000")
    assert bench.committed_traffic("joint") is None
    assert bench.committed_traffic("pooled4", "pooled") is None


def test_traffic_is_null_for_workloads_not_captured():
    assert bench.committed_traffic("named5") is None
    assert bench.committed_traffic("groups5", "pooled") is None


def test_algorithmic_flops():
    class P:
        count, width = 1000, 64
    assert bench.pooled_flops(P) == 3.0 * 1000 * 1000 * 64
    assert bench.pooled_flops(P, [16, 64]) == 3.0 * 1000 * 1000 * 80
