"""The synthetic workloads against the configuration the pages print (CPU).

tests/golden/ep_workload_shape.txt holds the expert-parallel shape of the
token-dispatch + GEMM figure; the ep, skew and decode workloads (and the
benchmark's metric) must use exactly that shape.
"""
import os

import pytest

import inputgen as ig

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "ep_workload_shape.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split()
                vals[key] = int(val)
    return vals


def test_golden_file_is_complete():
    assert set(_golden()) == {"top_k", "num_experts", "D", "D_expert"}


@pytest.mark.parametrize("name", ["ep", "skew", "decode"])
def test_workloads_use_the_printed_shape(name):
    g = _golden()
    wl = ig.WORKLOADS[name]
    assert (wl.k, wl.E, wl.D, wl.De) == (g["top_k"], g["num_experts"], g["D"], g["D_expert"])


def test_bench_metric_names_the_printed_shape():
    import bench
    g = _golden()
    assert f"D={g['D']}" in bench.METRIC and f"E={g['num_experts']}" in bench.METRIC
    assert f"k={g['top_k']}" in bench.METRIC
