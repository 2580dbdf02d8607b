"""Regression guard: the oracle on the tiny_f32 workload still produces the
values stored in tests/golden/tiny_f32_oracle.txt (written by
tests/golden/make_golden.py, which calls only oracle/).  The tolerance allows
for last-bit differences of the host libm between machines."""
import os
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_oracle_matches_stored_values():
    stored = {}
    with open(os.path.join(HERE, "golden", "tiny_f32_oracle.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split()
            stored[k] = float(v)
    now = make_golden.compute()
    assert set(now) == set(stored)
    for k, v in stored.items():
        assert now[k] == pytest.approx(v, rel=1e-5, abs=1e-6), k
