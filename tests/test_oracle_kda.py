"""Pins of the oracle's KDA recurrence (O6), [cpu_ops.cpp] KdaHeadTokenStep /
KdaGatedDeltaRuleKernel: the gated delta rule with one log decay per key
channel, g [T, Hv, Dk], q and k used as given.

Each pin checks a fact that does not re-type the recurrence:
  * a decay that is the same on every key channel is the plain gated delta
    rule: the KDA chain then equals the GDN oracle (itself pinned) bit for bit;
  * one token from a zero state has the closed form out = beta v (k.q) scale and
    leaves S = beta v k^T;
  * permuting the key channels of q, k, g and of the state's columns leaves the
    outputs unchanged and permutes the final state's columns (each channel's
    decay travels with it);
  * a channel whose decay is e^{-inf} forgets its column: after it, the state's
    column is that token's rank-1 update alone;
  * the f32 instantiation tracks f64;
  * the chunked form (O9) equals the token-by-token recurrence for any chunk
    length, with ragged tails, padding, fresh states and decays down to
    e^{-30} per token and channel; with one decay for every channel it is the
    GDN chunked form (O4, itself pinned).
"""
import numpy as np
import pytest

import oracle


def _inputs(seed, seqs=(5, 1, 9), Hk=2, Hv=4, Dk=16, Dv=8, slots=5):
    r = np.random.default_rng(seed)
    T = sum(seqs)
    cu = np.concatenate([[0], np.cumsum(seqs)]).astype(np.int32)
    q = r.normal(size=(T, Hk, Dk)) * 0.3
    k = r.normal(size=(T, Hk, Dk)) * 0.3
    v = r.normal(size=(T, Hv, Dv))
    g = -r.uniform(0.01, 2.0, size=(T, Hv, Dk))
    beta = r.uniform(0.1, 0.9, size=(T, Hv))
    pool = r.normal(size=(slots, Hv, Dv, Dk)) * 0.1
    sidx = np.array([3, 0, 4][:len(seqs)], np.int32)
    return q, k, v, g, beta, pool, cu, sidx


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_uniform_channel_decay_is_gdn(dtype):
    q, k, v, g, beta, pool, cu, sidx = _inputs(1)
    g_head = g[:, :, 0]
    g_uniform = np.repeat(g_head[:, :, None], g.shape[2], axis=2)
    p1, p2 = pool.astype(dtype), pool.astype(dtype)
    a = oracle.kda_varlen(q, k, v, g_uniform, beta, p1, cu, 0.25, state_indices=sidx, dtype=dtype)
    b = oracle.gdn_varlen(q, k, v, g_head, beta, p2, cu, 0.25, state_indices=sidx, dtype=dtype)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(p1, p2)


def test_one_token_closed_form():
    r = np.random.default_rng(2)
    Dk, Dv = 8, 4
    q, k = r.normal(size=(1, 1, Dk)), r.normal(size=(1, 1, Dk))
    v = r.normal(size=(1, 1, Dv))
    g = -r.uniform(0, 3, size=(1, 1, Dk))
    beta = np.array([[0.625]])
    pool = np.zeros((1, 1, Dv, Dk))
    out = oracle.kda_varlen(q, k, v, g, beta, pool, [0, 1], 0.5, dtype=np.float64)
    np.testing.assert_allclose(out[0, 0], 0.625 * v[0, 0] * (k[0, 0] @ q[0, 0]) * 0.5, rtol=1e-13)
    np.testing.assert_allclose(pool[0, 0], 0.625 * np.outer(v[0, 0], k[0, 0]), rtol=1e-13)


def test_key_channel_permutation():
    q, k, v, g, beta, pool, cu, sidx = _inputs(3)
    perm = np.random.default_rng(4).permutation(q.shape[2])
    p1, p2 = pool.copy(), pool[..., perm].copy()
    a = oracle.kda_varlen(q, k, v, g, beta, p1, cu, 0.3, state_indices=sidx, dtype=np.float64)
    b = oracle.kda_varlen(q[..., perm], k[..., perm], v, g[..., perm], beta, p2, cu, 0.3,
                          state_indices=sidx, dtype=np.float64)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(p1[..., perm], p2, rtol=1e-12, atol=1e-14)


def test_full_forgetting_channel():
    q, k, v, g, beta, pool, cu, sidx = _inputs(5, seqs=(6,), slots=1)
    sidx = np.array([0], np.int32)
    d0, t_last = 3, 5
    g = g.copy()
    g[t_last, :, d0] = -np.inf  # e^{-inf} = 0: column d0 forgets everything before t_last
    p = pool.copy()
    oracle.kda_varlen(q, k, v, g, beta, p, cu, 0.3, state_indices=sidx, dtype=np.float64)
    # the row's dot with k before the update uses the decayed row; column d0 of
    # the final state is then exactly the last token's update u_i k_{d0}
    p_before = pool.copy()
    oracle.kda_varlen(q[:t_last], k[:t_last], v[:t_last], g[:t_last], beta[:t_last], p_before,
                      [0, t_last], 0.3, state_indices=sidx, dtype=np.float64)
    hk = np.arange(v.shape[1]) // (v.shape[1] // q.shape[1])
    for h in range(v.shape[1]):
        decayed = p_before[0, h] * np.exp(g[t_last, h])[None, :]
        u = beta[t_last, h] * (v[t_last, h] - decayed @ k[t_last, hk[h]])
        np.testing.assert_allclose(p[0, h][:, d0], u * k[t_last, hk[h], d0], rtol=1e-12,
                                   atol=1e-15)


def test_f32_tracks_f64():
    q, k, v, g, beta, pool, cu, sidx = _inputs(6, Dk=64, Dv=32)
    p1, p2 = pool.astype(np.float64), pool.astype(np.float32)
    a = oracle.kda_varlen(q, k, v, g, beta, p1, cu, 0.2, state_indices=sidx, dtype=np.float64)
    b = oracle.kda_varlen(q, k, v, g, beta, p2, cu, 0.2, state_indices=sidx, dtype=np.float32)
    assert np.abs(a - b).max() / np.sqrt((a ** 2).mean()) < 1e-5


@pytest.mark.parametrize("chunk", [1, 7, 16, 64])
@pytest.mark.parametrize("strong", [False, True])
def test_chunked_form_equals_recurrence(chunk, strong):
    q, k, v, g, beta, pool, cu, sidx = _inputs(7 + chunk, seqs=(5, 1, 70, 33))
    sidx = np.array([3, -1, 0, 4], np.int32)
    has_init = np.array([1, 1, 0, 1], np.uint8)
    if strong:
        g = -np.random.default_rng(11).uniform(0.0, 30.0, size=g.shape)
    p1, p2 = pool.copy(), pool.copy()
    a = oracle.kda_varlen(q, k, v, g, beta, p1, cu, 0.3, state_indices=sidx,
                          has_initial_state=has_init, dtype=np.float64)
    b = oracle.kda_chunked_f64(q, k, v, g, beta, p2, cu, 0.3, chunk, state_indices=sidx,
                               has_initial_state=has_init)
    scale_o = np.sqrt((a ** 2).mean())
    assert np.abs(a - b).max() <= 1e-10 * scale_o
    assert np.abs(p1 - p2).max() <= 1e-10 * np.sqrt((p1 ** 2).mean())


def test_chunked_form_with_uniform_decay_is_gdn_chunked():
    q, k, v, g, beta, pool, cu, sidx = _inputs(9, seqs=(40, 3))
    g_head = g[:, :, 0]
    g_uniform = np.repeat(g_head[:, :, None], g.shape[2], axis=2)
    p1, p2 = pool.copy(), pool.copy()
    a = oracle.kda_chunked_f64(q, k, v, g_uniform, beta, p1, cu, 0.25, 16, state_indices=sidx)
    b = oracle.gdn_chunked_f64(q, k, v, g_head, beta, p2, cu, 0.25, 16, state_indices=sidx)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(p1, p2, rtol=1e-11, atol=1e-13)
