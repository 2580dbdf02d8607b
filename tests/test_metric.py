"""The bf16-storage parity metric of tests/helpers.py: exact rounding of the
reference scores 0, a one-quantum rounding flip scores 0, and anything beyond
one quantum counts in full."""
import numpy as np
import pytest

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


def test_bf16_flip_finds_the_neighbour_across_the_boundary():
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7: rounds to even (1), neighbour above
    r, nb, d = H.bf16_flip(np.array([1 + 2.0 ** -8]))
    assert (r[0], nb[0], d[0]) == (1.0, 1 + 2.0 ** -7, 0.0)
    # just below 1 the spacing halves: the neighbour is 1 - 2^-8, the boundary 1 - 2^-9
    r, nb, d = H.bf16_flip(np.array([1 - 2.0 ** -10]))
    assert (r[0], nb[0], d[0]) == (1.0, 1 - 2.0 ** -8, 2.0 ** -10)
    # negative values mirror it; exact bf16 values and zero have no neighbour to flip to
    r, nb, d = H.bf16_flip(np.array([-(1 + 2.0 ** -8 + 2.0 ** -12), -3.0, 0.0]))
    assert r[0] == -(1 + 2.0 ** -7) and nb[0] == -1.0 and d[0] == 2.0 ** -12
    assert nb[1] == r[1] == -3.0 and nb[2] == r[2] == 0.0


def _prepared(weak, seed, D=16, seqlens=(70, 1, 130)):
    import torch
    from gated_delta_rule_44_gb300 import workloads as W
    w = W.make_workload("flip", seed, list(seqlens), 1, 2, D, D, act_dtype=torch.float32,
                        weak_decay=weak, state_std=0.3, slots=len(seqlens) + 2)
    prep, _ = H.oracle_prepare(w)
    return w, {k: v.astype(np.float64) for k, v in prep.items()}


def _run(w, prep, with_pool=False, **over):
    import oracle
    x = dict(prep, **over)
    pool = w.state_pool.numpy().astype(np.float64).copy()
    out = oracle.gdn_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], pool,
                            w.cu_seqlens.numpy(), 1.0 / np.sqrt(w.Dk),
                            state_indices=w.state_indices.numpy(),
                            has_initial_state=w.has_initial_state.numpy(), dtype=np.float64)
    return (out, pool) if with_pool else out


@pytest.mark.parametrize("weak", [False, True])
@pytest.mark.parametrize("which", ["q", "k", "v", "qkv"])
def test_deviation_bound_holds_and_is_tight(weak, which):
    """Moving stored q, k or v values (3 % of them, each by up to its bf16
    step) moves the oracle's outputs by no more than the oracle's first-order
    deviation bound (with 1 % for second-order terms), and the bound is within
    a small factor of the largest move actually seen."""
    import oracle
    w, prep = _prepared(weak, 61 + weak, D=64, seqlens=(70, 1, 130))
    rng = np.random.default_rng(7 + weak)
    moves, over = {}, {}
    for key in ("q", "k", "v"):
        x = prep[key]
        step = np.abs(H.bf16_flip(x)[1] - H.bf16_round(x)) + np.abs(x) * 2.0 ** -8
        m = np.where(rng.random(x.shape) < 0.03, step, 0.0) if key in which else np.zeros_like(x)
        moves[key] = m
        over[key] = x + m * rng.choice([-1.0, 1.0], size=x.shape)
    o1, s1 = _run(w, prep, with_pool=True)
    o2, s2 = _run(w, prep, with_pool=True, **over)
    bound, sbound = oracle.gdn_deviation_bound(
        prep["q"], prep["k"], prep["v"], prep["g"], prep["beta"], moves["q"], moves["k"],
        moves["v"], w.state_pool.numpy().astype(np.float64), w.cu_seqlens.numpy(),
        1.0 / np.sqrt(w.Dk), state_indices=w.state_indices.numpy(),
        has_initial_state=w.has_initial_state.numpy(), with_state=True)
    moved = np.abs(o2 - o1)
    assert np.all(moved <= bound * 1.01 + 1e-15)
    live = bound > 1e-12
    assert (moved[live] / bound[live]).max() > 0.2
    # the final states: every element of a row within the row's bound
    smoved = np.abs(s2 - s1)
    assert np.all(smoved <= sbound[..., None] * 1.01 + 1e-15)
    if which != "q":  # q does not enter the state
        rows = sbound > 1e-12
        assert (smoved.max(axis=-1)[rows] / sbound[rows]).max() > 0.05


def test_deviation_bound_is_zero_without_moves_and_linear_in_them():
    import oracle
    w, prep = _prepared(True, 65)
    z = np.zeros_like(prep["q"])
    args = (prep["q"], prep["k"], prep["v"], prep["g"], prep["beta"])
    kw = dict(state_indices=w.state_indices.numpy(), has_initial_state=w.has_initial_state.numpy())
    pool = w.state_pool.numpy().astype(np.float64)
    zero = oracle.gdn_deviation_bound(*args, z, z, np.zeros_like(prep["v"]), pool,
                                      w.cu_seqlens.numpy(), 0.25, **kw)
    assert not zero.any()
    dv = np.full_like(prep["v"], 1e-3)
    b1 = oracle.gdn_deviation_bound(*args, z, z, dv, pool, w.cu_seqlens.numpy(), 0.25, **kw)
    b2 = oracle.gdn_deviation_bound(*args, z, z, 2 * dv, pool, w.cu_seqlens.numpy(), 0.25, **kw)
    assert np.allclose(b2, 2 * b1) and b1.min() > 0
