"""The committed ncu records that bench.py reads (no GPU needed).

bench.py reports a GEMM's per-launch DRAM traffic only while the GEMM
sources hash to the build the counters were taken on; these checks keep the
records and the sources in step, and each record's figures consistent.
"""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RECORDS = ["lm_head_gemm_traffic.json", "gate_up_gemm_traffic.json", "lm_head_gemm_shortlist_traffic.json"]


def _bench():
    spec = importlib.util.spec_from_file_location("bench_for_profiles", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("record", RECORDS)
def test_traffic_record_matches_the_gemm_sources(record):
    bench = _bench()
    with open(os.path.join(ROOT, "profiles", record)) as f:
        d = json.load(f)
    assert d["kernel_source_hash"] == bench.head_kernel_hash(), (
        f"{record} was taken on other GEMM sources: capture the counters again")
    assert d["dram_bytes_per_launch"] == d["dram_bytes_read"] + d["dram_bytes_write"]
    # DRAM traffic near the algorithmic bytes: the weights stream once per launch
    assert 0.9 <= d["dram_bytes_per_launch"] / d["algorithmic_bytes_per_launch"] <= 1.1
    assert d["command"].startswith("ncu ") and "--clock-control none" in d["command"]
    assert bench.recorded_traffic(d["workload"], d["rows"], record) == d["dram_bytes_per_launch"]


def test_traffic_is_withheld_for_another_workload():
    bench = _bench()
    assert bench.recorded_traffic("no-such-workload", 1024) is None
