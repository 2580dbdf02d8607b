"""Pins of the oracle's gated RMSNorm (O5), [cpu.rs] gated_rms_norm_f32 with
[cpu_ops.cpp] RmsNormGatedKernel's sigmoid gate and strided gate rows.

Each pin checks a fact that does not re-type the formula:
  * with eps = 0 every row of out / (weight * act(z)) has root-mean-square 1
    (the normalisation divides by the mean, not the sum, of squares);
  * scaling a row of core by any alpha > 0 leaves the output unchanged (eps = 0);
  * a constant row c with eps e is scaled by c / sqrt(c^2 + e): c = 3, e = 7
    gives 3/4; z = ln 3 makes the sigmoid exactly 3/4, so silu(ln 3) = 0.75 ln 3;
  * the sigmoid gate of z = 0 is 1/2 and its silu is 0;
  * a gate given as wider token rows (a merged projection's slice) equals the
    same values given contiguously;
  * a row depends on its own (token, head) only;
  * the f32 instantiation tracks the f64 one;
  * the validator's messages are the page's (validate_gated_rms_norm_shape).
"""
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _inputs(seed, T=5, H=3, D=16):
    r = np.random.default_rng(seed)
    core = r.normal(size=(T, H, D))
    z = r.uniform(1.0, 3.0, size=(T, H, D))      # act(z) well away from 0
    w = r.uniform(0.5, 2.0, size=D)
    return core, z, w


def _act(z, sigmoid_gate):
    s = 1.0 / (1.0 + np.exp(-z))
    return s if sigmoid_gate else z * s


@pytest.mark.parametrize("sigmoid_gate", [False, True])
def test_unit_rms_without_eps(sigmoid_gate):
    core, z, w = _inputs(1)
    out = oracle.gated_rmsnorm(core, z, w, 0.0, sigmoid_gate=sigmoid_gate)
    normed = out / (w * _act(z, sigmoid_gate))
    rms = np.sqrt((normed ** 2).mean(axis=-1))
    np.testing.assert_allclose(rms, 1.0, rtol=1e-12)


def test_scale_invariance_without_eps():
    core, z, w = _inputs(2)
    alpha = np.random.default_rng(3).uniform(0.01, 100.0, size=core.shape[:2] + (1,))
    a = oracle.gated_rmsnorm(core, z, w, 0.0)
    b = oracle.gated_rmsnorm(core * alpha, z, w, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=0)


def test_constant_row_closed_form():
    D = 8
    core = np.full((1, 1, D), 3.0)
    z = np.full((1, 1, D), math.log(3.0))
    w = np.arange(1, D + 1, dtype=np.float64)
    out = oracle.gated_rmsnorm(core, z, w, 7.0)
    # 3 / sqrt(9 + 7) = 3/4;  silu(ln 3) = ln 3 * 3/4
    np.testing.assert_allclose(out[0, 0], 0.75 * w * 0.75 * math.log(3.0), rtol=1e-14)
    out_s = oracle.gated_rmsnorm(core, z, w, 7.0, sigmoid_gate=True)
    np.testing.assert_allclose(out_s[0, 0], 0.75 * w * 0.75, rtol=1e-14)


def test_gate_at_zero():
    core, _, w = _inputs(4)
    z = np.zeros_like(core)
    assert np.all(oracle.gated_rmsnorm(core, z, w, 1e-6) == 0.0)
    half = oracle.gated_rmsnorm(core, z, w, 0.0, sigmoid_gate=True)
    np.testing.assert_allclose(np.sqrt(((half / (w * 0.5)) ** 2).mean(axis=-1)), 1.0, rtol=1e-12)


def test_strided_gate_rows():
    core, z, w = _inputs(5)
    T, H, D = core.shape
    wide = np.random.default_rng(6).normal(size=(T, H * D + 24)) * 1e3  # garbage in the pad
    wide[:, :H * D] = z.reshape(T, H * D)
    np.testing.assert_array_equal(oracle.gated_rmsnorm(core, wide, w, 1e-6),
                                  oracle.gated_rmsnorm(core, z, w, 1e-6))


def test_rows_independent():
    core, z, w = _inputs(7)
    a = oracle.gated_rmsnorm(core, z, w, 1e-6)
    core2, z2 = core.copy(), z.copy()
    core2[2, 1] *= -5.0
    z2[2, 1] += 1.0
    b = oracle.gated_rmsnorm(core2, z2, w, 1e-6)
    mask = np.ones(core.shape[:2], bool)
    mask[2, 1] = False
    np.testing.assert_array_equal(a[mask], b[mask])
    assert not np.allclose(a[2, 1], b[2, 1])


def test_f32_tracks_f64():
    core, z, w = _inputs(8, T=40, H=4, D=128)
    a = oracle.gated_rmsnorm(core, z, w, 1e-6, dtype=np.float64)
    b = oracle.gated_rmsnorm(core, z, w, 1e-6, dtype=np.float32)
    assert np.abs(a - b).max() / np.sqrt((a ** 2).mean()) < 1e-5


def test_validator_messages():
    rc, msg = oracle.validate_gated_rms_norm_shape(48, 48, 8, 48, 3, 0, 8)
    assert rc != 0 and msg == "gated_rms_norm shape must be positive, got tokens=3 heads=0 dim=8"
    for lens, label, actual in (((47, 48, 8, 48), "core", 47), ((48, 40, 8, 48), "z", 40),
                                ((48, 48, 7, 48), "weight", 7), ((48, 48, 8, 1), "out", 1)):
        rc, msg = oracle.validate_gated_rms_norm_shape(*lens, 3, 2, 8)
        expected = 8 if label == "weight" else 48
        assert rc != 0 and msg == f"gated_rms_norm {label} length {actual} < expected {expected}"
    assert oracle.validate_gated_rms_norm_shape(48, 48, 8, 48, 3, 2, 8) == (0, "")
