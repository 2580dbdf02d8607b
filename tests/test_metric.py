"""The bf16-storage parity metric of tests/helpers.py: exact rounding of the
reference scores 0, a one-quantum rounding flip scores 0, and anything beyond
one quantum counts in full."""
import numpy as np

import helpers as H


def test_rounded_reference_scores_zero():
    rng = np.random.default_rng(0)
    ref = rng.standard_t(3, size=10000) * 5  # heavy tails
    assert H.rel_err_stored_bf16(H.bf16_round(ref), ref) == 0.0
    assert H.rel_err(H.bf16_round(ref), ref) > 1e-3  # the plain metric sees the rounding


def test_one_quantum_flip_is_exempt_two_are_not():
    ref = np.array([1.0, 3.0, -0.75, 100.0])
    rq = H.bf16_round(ref)
    q = H.bf16_quantum(rq)
    assert np.allclose(q, [2.0 ** -7, 2.0 ** -6, 2.0 ** -8, 2.0 ** -1])
    assert H.rel_err_stored_bf16(rq + q, ref) == 0.0
    rms = np.sqrt((ref ** 2).mean())
    got = rq.copy()
    got[3] += 3 * q[3]
    assert np.isclose(H.rel_err_stored_bf16(got, ref), 2 * q[3] / rms)
