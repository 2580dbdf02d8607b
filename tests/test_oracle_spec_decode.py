"""Pins of the oracle's speculative multi-token decode (O7), [cpu_ops.cpp]
GdnSpecDecodeKernel: each request runs its draft tokens through the gated
delta rule from the snapshot of its last accepted token, and stores the state
after every draft token in its own slot so that a later step can roll back to
any of them.

Each pin checks a fact that the page states or the mathematics fixes:
  * rollback: the snapshot after draft token j equals the state that the plain
    recurrence (the GDN oracle, itself pinned) reaches over the first j + 1
    tokens alone, bit for bit, and the outputs equal that recurrence's;
  * the initial state is the slot in column num_accepted - 1, whatever the
    other columns hold;
  * a negative initial slot zeroes that request's outputs and leaves the pool
    alone, a negative column skips only its own store, an empty request does
    nothing;
  * a tiny case matches a brute-force recurrence written with outer products;
  * malformed metadata (num_accepted outside [1, num_cols], a request longer
    than its row, a slot past the pool) is rejected;
  * the f32 instantiation tracks f64.
"""
import numpy as np
import pytest

import oracle


def _inputs(seed, lens=(3, 4, 1), Hk=2, Hv=4, Dk=16, Dv=8, num_cols=4, slots=16):
    r = np.random.default_rng(seed)
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = r.normal(size=(T, Hk, Dk)) * 0.3
    k = r.normal(size=(T, Hk, Dk)) * 0.3
    v = r.normal(size=(T, Hv, Dv))
    g = -r.uniform(0.01, 2.0, size=(T, Hv))
    beta = r.uniform(0.1, 0.9, size=(T, Hv))
    pool = r.normal(size=(slots, Hv, Dv, Dk)) * 0.1
    # each request owns a disjoint row of distinct slots
    sidx = r.permutation(slots)[:len(lens) * num_cols].reshape(len(lens), num_cols)
    nat = r.integers(1, num_cols + 1, size=len(lens))
    return q, k, v, g, beta, pool, cu, sidx.astype(np.int32), nat.astype(np.int32)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_rollback_equals_prefix_recurrence(dtype):
    q, k, v, g, beta, pool, cu, sidx, nat = _inputs(1)
    p = pool.astype(dtype)
    out = oracle.gdn_spec_decode(q, k, v, g, beta, p, cu, sidx, nat, 0.25, dtype=dtype)
    for i in range(len(nat)):
        lo, hi = cu[i], cu[i + 1]
        init = sidx[i, nat[i] - 1]
        for j in range(hi - lo):
            ref_pool = pool[[init]].astype(dtype)
            ref_out = oracle.gdn_varlen(q[lo:lo + j + 1], k[lo:lo + j + 1], v[lo:lo + j + 1],
                                        g[lo:lo + j + 1], beta[lo:lo + j + 1], ref_pool,
                                        [0, j + 1], 0.25, state_indices=[0], dtype=dtype)
            np.testing.assert_array_equal(p[sidx[i, j]], ref_pool[0])
            np.testing.assert_array_equal(out[lo:lo + j + 1], ref_out)


def test_initial_slot_is_column_of_last_accepted():
    q, k, v, g, beta, pool, cu, sidx, _ = _inputs(2, lens=(2,), num_cols=4)
    outs = []
    for n in range(1, 5):
        p = pool.copy()
        outs.append(oracle.gdn_spec_decode(q, k, v, g, beta, p, cu, sidx, [n], 0.3,
                                           dtype=np.float64))
        ref = pool[[sidx[0, n - 1]]].copy()
        want = oracle.gdn_varlen(q, k, v, g, beta, ref, cu, 0.3, state_indices=[0],
                                 dtype=np.float64)
        np.testing.assert_array_equal(outs[-1], want)
    # four different initial states give four different outputs
    assert len({o.tobytes() for o in outs}) == 4


def test_null_initial_slot_and_null_columns():
    q, k, v, g, beta, pool, cu, sidx, nat = _inputs(3, lens=(3, 3, 0, 2))
    sidx[0, nat[0] - 1] = -1          # request 0: no initial state
    nat[1] = 4                        # request 1 starts from column 3 ...
    sidx[1, 1] = -5                   # ... and skips the store after its token 1
    p = pool.copy()
    out = np.full((q.shape[0], v.shape[1], v.shape[2]), 7.0)
    oracle.gdn_spec_decode(q, k, v, g, beta, p, cu, sidx, nat, 0.3, out=out, dtype=np.float64)
    assert not out[cu[0]:cu[1]].any()
    # the skipped store changes nothing downstream: request 1's outputs and its
    # other snapshots are those of the plain recurrence from its initial slot
    lo, hi = cu[1], cu[2]
    ref_pool = pool[[sidx[1, 3]]].copy()
    want = oracle.gdn_varlen(q[lo:hi], k[lo:hi], v[lo:hi], g[lo:hi], beta[lo:hi], ref_pool,
                             [0, hi - lo], 0.3, state_indices=[0], dtype=np.float64)
    np.testing.assert_array_equal(out[lo:hi], want)
    np.testing.assert_array_equal(p[sidx[1, 2]], ref_pool[0])
    written = set()
    for i in (1, 3):
        for j in range(cu[i + 1] - cu[i]):
            if sidx[i, j] >= 0:
                written.add(int(sidx[i, j]))
    for s_ in range(pool.shape[0]):
        if s_ not in written:
            np.testing.assert_array_equal(p[s_], pool[s_])
    # the empty request 2 owns no output row and writes no slot
    assert (out[cu[3]:] != 7.0).all() and (out[cu[1]:cu[2]] != 7.0).all()


def test_brute_force_tiny():
    q, k, v, g, beta, pool, cu, sidx, nat = _inputs(4, lens=(3,), Hk=1, Hv=2, Dk=3, Dv=2,
                                                    num_cols=3, slots=4)
    scale = 0.7
    p = pool.copy()
    out = oracle.gdn_spec_decode(q, k, v, g, beta, p, cu, sidx, nat, scale, dtype=np.float64)
    for h in range(2):
        S = pool[sidx[0, nat[0] - 1], h].copy()
        for t in range(3):
            S = S * np.exp(g[t, h])
            S = S + np.outer(beta[t, h] * (v[t, h] - S @ k[t, 0]), k[t, 0])
            np.testing.assert_allclose(out[t, h], S @ (scale * q[t, 0]), rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(p[sidx[0, t], h], S, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("case", ["nat0", "nat_big", "too_long", "slot_big"])
def test_rejects_bad_metadata(case):
    q, k, v, g, beta, pool, cu, sidx, nat = _inputs(5, lens=(3, 2), num_cols=3)
    if case == "nat0":
        nat[0] = 0
    elif case == "nat_big":
        nat[1] = 4
    elif case == "too_long":
        cu = np.array([0, 1, 5], np.int32)   # request 1 has 4 tokens, its row has 3
    else:
        sidx[1, 2] = pool.shape[0]
    with pytest.raises(oracle.OracleError):
        oracle.gdn_spec_decode(q, k, v, g, beta, pool.copy(), cu, sidx, nat, 0.3,
                               dtype=np.float64)


def test_f32_tracks_f64():
    q, k, v, g, beta, pool, cu, sidx, nat = _inputs(6, Dk=64, Dv=32)
    p1, p2 = pool.astype(np.float64), pool.astype(np.float32)
    a = oracle.gdn_spec_decode(q, k, v, g, beta, p1, cu, sidx, nat, 0.2, dtype=np.float64)
    b = oracle.gdn_spec_decode(q, k, v, g, beta, p2, cu, sidx, nat, 0.2, dtype=np.float32)
    assert np.abs(a - b).max() / np.sqrt((a ** 2).mean()) < 1e-5
    assert np.abs(p1 - p2).max() / np.sqrt((p1 ** 2).mean()) < 1e-5
