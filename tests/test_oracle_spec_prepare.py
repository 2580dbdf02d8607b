"""Pins of the oracle's speculative prepare (O8), [cpu_ops.cpp]
CausalConv1dSpecUpdateKernel: the causal conv of the prepare step for the
draft tokens of a speculative step, on a widened conv row of
(K-1) + (max_q - 1) raw inputs read at offset num_accepted - 1.

Each pin checks a fact that the page states or the mathematics fixes:
  * with one draft per request and max_q = 1 the widened row is the plain
    K-1 tail, and the step equals the decode prepare (O1, itself pinned) bit
    for bit, gates and norm included;
  * over a run of speculative steps, each accepting a random prefix of its
    drafts, every draft's conv output is the plain causal convolution
    (numpy.convolve) of the accepted history followed by the drafts so far;
    this is what the one-tap shift and the offset are for;
  * a negative slot gives the outputs of a zero window and writes no row; an
    empty request does nothing;
  * malformed metadata is rejected; the f32 instantiation tracks f64.
"""
import numpy as np
import pytest

import oracle

Hk, Hv, Dk, Dv, K = 1, 2, 8, 4, 4
C = 2 * Hk * Dk + Hv * Dv


def _common(r, T):
    x = r.normal(size=(T, C))
    w = r.normal(size=(C, K)) * 0.5
    a = r.normal(size=(T, Hv))
    b = r.normal(size=(T, Hv))
    A_log = r.normal(size=Hv) * 0.3
    dt_bias = r.normal(size=Hv) * 0.3
    return x, w, a, b, A_log, dt_bias


def _silu(z):
    return z / (1.0 + np.exp(-z))


def test_single_draft_is_decode_prepare():
    r = np.random.default_rng(1)
    n = 5
    x, w, a, b, A_log, dt_bias = _common(r, n)
    pool = r.normal(size=(7, C, K - 1))
    idx = np.array([3, 0, -1, 6, 2], np.int32)
    cu = np.arange(n + 1, dtype=np.int32)
    p1, p2 = pool.copy(), pool.copy()
    got = oracle.spec_prepare(x, w, p1, a, b, A_log, dt_bias, cu, idx, np.ones(n, np.int32),
                              Hk, Hv, Dk, Dv, K, dtype=np.float64)
    want = oracle.prepare_varlen(x, w, p2, a, b, A_log, dt_bias, cu, Hk, Hv, Dk, Dv, K,
                                 state_indices=idx, dtype=np.float64)
    for name in ("q", "k", "v", "g", "beta"):
        np.testing.assert_array_equal(got[name], want[name], err_msg=name)
    np.testing.assert_array_equal(p1, p2)


@pytest.mark.parametrize("max_q", [1, 2, 4, 6])
def test_outputs_are_the_convolution_of_the_accepted_history(max_q):
    r = np.random.default_rng(10 + max_q)
    n_reqs, steps, W = 3, 5, K - 1
    w = r.normal(size=(C, K)) * 0.5
    A_log, dt_bias = np.zeros(Hv), np.zeros(Hv)
    pool = np.zeros((n_reqs, C, W + max_q - 1))
    idx = np.arange(n_reqs, dtype=np.int32)[::-1].copy()
    history = [np.zeros((W, C)) for _ in range(n_reqs)]   # the zero row is a zero past
    nat = np.ones(n_reqs, np.int32)
    for _ in range(steps):
        drafts = r.normal(size=(n_reqs * max_q, C))
        cu = np.arange(0, n_reqs * max_q + 1, max_q, dtype=np.int32)
        zeros = np.zeros((n_reqs * max_q, Hv))
        out = oracle.spec_prepare(drafts, w, pool, zeros, zeros, A_log, dt_bias, cu, idx, nat,
                                  Hk, Hv, Dk, Dv, K, apply_qk_l2norm=False, dtype=np.float64)
        flat = np.concatenate([out["q"].reshape(len(drafts), -1), out["k"].reshape(len(drafts), -1),
                               out["v"].reshape(len(drafts), -1)], axis=1)
        for i in range(n_reqs):
            d = drafts[i * max_q:(i + 1) * max_q]
            seq = np.concatenate([history[i], d])
            for c in range(C):
                full = np.convolve(seq[:, c], w[c, ::-1])   # causal: sum_j w[j] x[t-W+j]
                want = _silu(full[len(history[i]):len(seq)])
                np.testing.assert_allclose(flat[i * max_q:(i + 1) * max_q, c], want,
                                           rtol=1e-12, atol=1e-14)
        # the verifier accepts a random prefix of each request's drafts
        nat = r.integers(1, max_q + 1, size=n_reqs).astype(np.int32)
        for i in range(n_reqs):
            history[i] = np.concatenate([history[i], drafts[i * max_q:i * max_q + nat[i]]])


def test_null_slot_and_empty_request():
    r = np.random.default_rng(3)
    lens, max_q = (2, 0, 3), 3
    T = sum(lens)
    x, w, a, b, A_log, dt_bias = _common(r, T)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pool = r.normal(size=(4, C, K - 1 + max_q - 1))
    p = pool.copy()
    idx = np.array([-1, 1, 2], np.int32)
    nat = np.array([2, 3, 1], np.int32)
    got = oracle.spec_prepare(x, w, p, a, b, A_log, dt_bias, cu, idx, nat, Hk, Hv, Dk, Dv, K,
                              apply_qk_l2norm=False, dtype=np.float64)
    # request 0 has no row: a zero window, i.e. the plain conv of its drafts alone
    v0 = got["v"][:2].reshape(2, -1)
    for c in range(2 * Hk * Dk, C):
        want = _silu(np.convolve(x[:2, c], w[c, ::-1])[:2])
        np.testing.assert_allclose(v0[:, c - 2 * Hk * Dk], want, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(p[[0, 1, 3]], pool[[0, 1, 3]])   # only request 2's row moved
    assert not np.array_equal(p[2], pool[2])


@pytest.mark.parametrize("case", ["nat0", "nat_big", "too_long", "slot_big", "short_row", "k1"])
def test_rejects_bad_metadata(case):
    r = np.random.default_rng(4)
    max_q = 3
    lens = [3, 2]
    cu = np.array([0, 3, 5], np.int32)
    x, w, a, b, A_log, dt_bias = _common(r, 5)
    pool = np.zeros((3, C, K - 1 + max_q - 1))
    idx = np.array([0, 1], np.int32)
    nat = np.array([1, 3], np.int32)
    if case == "nat0":
        nat[0] = 0
    elif case == "nat_big":
        nat[1] = 4
    elif case == "too_long":
        cu = np.array([0, 4, 5], np.int32)
    elif case == "slot_big":
        idx[1] = 3
    elif case == "short_row":
        pool = np.zeros((3, C, K - 2))   # shorter than the K-1 tail
    kw = K
    if case == "k1":                     # no conv tail: nothing to carry
        kw, w = 1, w[:, :1]
    with pytest.raises(oracle.OracleError):
        oracle.spec_prepare(x, w, pool, a, b, A_log, dt_bias, cu, idx, nat, Hk, Hv, Dk, Dv, kw,
                            dtype=np.float64)


def test_f32_tracks_f64():
    r = np.random.default_rng(5)
    lens, max_q = (4, 4, 2, 4), 4
    T = sum(lens)
    x, w, a, b, A_log, dt_bias = _common(r, T)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pool = r.normal(size=(4, C, K - 1 + max_q - 1))
    idx = np.array([2, 0, 3, 1], np.int32)
    nat = np.array([1, 4, 2, 3], np.int32)
    p1, p2 = pool.astype(np.float64), pool.astype(np.float32)
    a64 = oracle.spec_prepare(x, w, p1, a, b, A_log, dt_bias, cu, idx, nat, Hk, Hv, Dk, Dv, K,
                              dtype=np.float64)
    a32 = oracle.spec_prepare(x, w, p2, a, b, A_log, dt_bias, cu, idx, nat, Hk, Hv, Dk, Dv, K,
                              dtype=np.float32)
    for name in ("q", "k", "v", "g", "beta"):
        ref = a64[name]
        assert np.abs(a32[name] - ref).max() / np.sqrt((ref ** 2).mean()) < 1e-5, name
    np.testing.assert_allclose(p2, p1, rtol=1e-6, atol=1e-7)
