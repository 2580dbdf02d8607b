"""Host-side logic of bench.py (no GPU): the roofline's measured DRAM traffic
applies only to the kernel source it was measured on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_matches_current_source():
    for (call, workload) in bench.MEASURED_TRAFFIC:
        nbytes, how = bench.measured_traffic(call, workload)
        assert (nbytes is None) == ("changed" in how), (call, workload, how)
        if nbytes is not None:
            assert nbytes > 0


def test_traffic_null_after_source_change(monkeypatch):
    table = dict(bench.MEASURED_TRAFFIC)
    key = ("prefill", "prefill_4k")
    b, src, sha, how = table[key]
    table[key] = (b, src, "0" * 64, how)
    monkeypatch.setattr(bench, "MEASURED_TRAFFIC", table)
    nbytes, reason = bench.measured_traffic(*key)
    assert nbytes is None and "changed" in reason
    assert bench.measured_traffic("prepare", "prefill_4k") == (None, "not captured")
