"""Pins of the oracle's gate functions against library routines.

[cpu.rs] (ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs) sigmoid,
silu and softplus.  Pins: sigmoid equals scipy.special.expit; softplus equals
numpy's logaddexp(0, x) = ln(1 + e^x) to the rounding of 1 + e^x (the pages switch to x above 20 and to
e^x below -20, both within 1e-8 of the exact value); silu(x) = x * expit(x);
the symmetry sigmoid(-x) = 1 - sigmoid(x); f32 and f64 instantiations agree.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle

XS = np.concatenate([np.linspace(-40, 40, 321), [-20.0, 20.0, -20.0001, 20.0001, 0.0, 1e-8,
                                                 -1e-8, 700.0, -700.0]])


def test_sigmoid_matches_expit():
    for x in XS:
        assert oracle.sigmoid(x) == pytest.approx(expit(x), rel=1e-14, abs=1e-300)


def test_sigmoid_symmetry():
    for x in XS:
        assert oracle.sigmoid(-x) == pytest.approx(1.0 - oracle.sigmoid(x), abs=1e-15)


def test_softplus_matches_logaddexp():
    for x in XS:
        exact = np.logaddexp(0.0, x)
        # ln(1 + e^x) loses the absolute precision of 1 + e^x (2.2e-16) below 0
        assert oracle.softplus(x) == pytest.approx(exact, rel=1e-8, abs=3e-16)


def test_softplus_branches():
    # identity above 20, exponential below -20 (the pages' thresholds)
    assert oracle.softplus(25.0) == 25.0
    assert oracle.softplus(-25.0) == np.exp(-25.0)
    assert oracle.softplus(0.0) == pytest.approx(np.log(2.0), rel=1e-15)


def test_silu_definition():
    for x in XS:
        assert oracle.silu(x) == pytest.approx(x * expit(x), rel=1e-14, abs=1e-300)


def test_f32_close_to_f64():
    for x in np.linspace(-30, 30, 121):
        for fn in (oracle.sigmoid, oracle.softplus, oracle.silu):
            a = fn(float(np.float32(x)), dtype=np.float32)
            b = fn(float(np.float32(x)), dtype=np.float64)
            # f32 ln(1 + e^x) rounds 1 + e^x to f32 (absolute error <= 6e-8)
            assert a == pytest.approx(b, rel=2e-6, abs=1.2e-7)
