"""Pins of the oracle's prepare step (O1) against library routines and identities.

Follows [cpu.rs] (ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs)
linear_attention_prepare_varlen_f32 / linear_attention_decode_prepare_batch_f32
and [cpu_ops.cpp] (vllm.cpp, src/vt/cpu/cpu_ops.cpp) CausalConv1dFwdKernel.
Pins, none of which re-types the oracle's loop:
  - pre-activation conv == numpy.convolve of (tail || x) with the reversed
    taps (a library convolution), SiLU via scipy.special.expit;
  - impulse response: a unit input at token t0 reproduces the taps, reversed,
    at t0..t0+K-1 (catches a reversed or shifted window);
  - new tail == the last K-1 entries of numpy.concatenate((tail, x));
  - q/k/v routing by channel range, GQA-independent;
  - gates == -exp(A_log) * logaddexp(0, a + dt_bias) and expit(b);
  - L2 norm: ||row|| == sqrt(ss / (ss + 1e-6)) in closed form;
  - split/resume with the tail carried == one run; a decode batch == each token
    alone; has_initial_state = 0 == zero tail; a -1 slot leaves the pool alone;
  - results do not depend on the thread count.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle

RNG = np.random.default_rng(1234)


def case(seqlens, Hk=2, Hv=4, Dk=4, Dv=3, K=4, slots=None, seed=0):
    rng = np.random.default_rng(seed)
    T = int(sum(seqlens))
    N = len(seqlens)
    C = 2 * Hk * Dk + Hv * Dv
    slots = slots or N
    d = dict(
        x=rng.normal(size=(T, C)), w=rng.normal(size=(C, K)) * 0.5,
        pool=rng.normal(size=(slots, C, K - 1)), a=rng.normal(size=(T, Hv)) * 2,
        b=rng.normal(size=(T, Hv)) * 2, alog=np.log(rng.uniform(1, 16, size=Hv)),
        dt=rng.normal(size=Hv) * 0.5,
        cu=np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32),
        Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K, T=T, N=N, C=C)
    return d


def run(d, pool=None, sidx=None, hinit=None, norm=False, dtype=np.float64, nthreads=0):
    pool = (d["pool"] if pool is None else pool).astype(dtype).copy()
    out = oracle.prepare_varlen(d["x"], d["w"], pool, d["a"], d["b"], d["alog"], d["dt"], d["cu"],
                                d["Hk"], d["Hv"], d["Dk"], d["Dv"], d["K"], state_indices=sidx,
                                has_initial_state=hinit, apply_qk_l2norm=norm, dtype=dtype,
                                nthreads=nthreads)
    return out, pool


def conv_outputs(out, d):
    T = d["T"]
    return np.concatenate([out["q"].reshape(T, -1), out["k"].reshape(T, -1),
                           out["v"].reshape(T, -1)], axis=1)


def test_conv_matches_numpy_convolve():
    d = case([7, 1, 12, 2, 3])
    out, _ = run(d)
    y = conv_outputs(out, d)
    K = d["K"]
    for s in range(d["N"]):
        lo, hi = d["cu"][s], d["cu"][s + 1]
        for c in range(d["C"]):
            ext = np.concatenate([d["pool"][s, c], d["x"][lo:hi, c]])
            acc = np.convolve(ext, d["w"][c, ::-1])[K - 1:K - 1 + (hi - lo)]
            np.testing.assert_allclose(y[lo:hi, c], acc * expit(acc), rtol=1e-12, atol=1e-14)


def test_impulse_response_reverses_taps():
    d = case([10], Hk=1, Hv=1, Dk=4, Dv=4, K=4)
    d["x"][:] = 0.0
    t0 = 3
    d["x"][t0, :] = 1.0
    out, _ = run(d, pool=np.zeros_like(d["pool"]))
    y = conv_outputs(out, d)
    for c in range(d["C"]):
        for t in range(d["T"]):
            lag = t - t0
            acc = d["w"][c, d["K"] - 1 - lag] if 0 <= lag < d["K"] else 0.0
            assert y[t, c] == pytest.approx(acc * expit(acc), abs=1e-15)


def test_new_tail_is_last_inputs():
    for L in (1, 2, 3, 4, 5, 9):
        d = case([L, 2], K=4)
        _, pool = run(d)
        for s in range(d["N"]):
            lo, hi = d["cu"][s], d["cu"][s + 1]
            for c in range(d["C"]):
                ext = np.concatenate([d["pool"][s, c], d["x"][lo:hi, c]])
                np.testing.assert_array_equal(pool[s, c], ext[-(d["K"] - 1):])


def test_slot_indices_and_padding():
    d = case([3, 2, 4], slots=6)
    sidx = np.array([4, -1, 1], np.int32)
    pool0 = RNG.normal(size=(6, d["C"], d["K"] - 1))
    out, pool = run(d, pool=pool0, sidx=sidx)
    # padded sequence: its outputs use a zero tail and no pool row is touched
    d2 = dict(d)
    d2["pool"] = np.stack([pool0[4], np.zeros_like(pool0[0]), pool0[1]])
    out2, pool2 = run(d2)
    for key in ("q", "k", "v", "g", "beta"):
        np.testing.assert_array_equal(out[key], out2[key])
    np.testing.assert_array_equal(pool[4], pool2[0])
    np.testing.assert_array_equal(pool[1], pool2[2])
    for untouched in (0, 2, 3, 5):
        np.testing.assert_array_equal(pool[untouched], pool0[untouched])


def test_has_initial_state_zero_means_zero_tail():
    d = case([5, 2])
    hinit = np.array([0, 1], np.uint8)
    out, pool = run(d, hinit=hinit)
    d0 = dict(d)
    p0 = d["pool"].copy()
    p0[0] = 0.0
    d0["pool"] = p0
    out0, pool0 = run(d0)
    for key in ("q", "k", "v"):
        np.testing.assert_array_equal(out[key], out0[key])
    np.testing.assert_array_equal(pool, pool0)  # the new tail is still written


def test_gates_match_library():
    d = case([6, 5], Hv=5)
    d["a"][0, 0] = 30.0   # identity branch of softplus
    d["a"][1, 1] = -40.0  # exponential branch
    out, _ = run(d)
    sp = np.logaddexp(0.0, d["a"] + d["dt"][None, :])
    np.testing.assert_allclose(out["g"], -np.exp(d["alog"])[None, :] * sp, rtol=1e-8,
                               atol=3e-15)
    np.testing.assert_allclose(out["beta"], expit(d["b"]), rtol=1e-14)
    assert np.all(out["g"] < 0) and np.all((out["beta"] > 0) & (out["beta"] < 1))


def test_l2_norm_closed_form():
    d = case([9], Hk=3, Dk=8)
    raw, _ = run(d, norm=False)
    nrm, _ = run(d, norm=True)
    for key in ("q", "k"):
        ss = (raw[key] ** 2).sum(-1)
        np.testing.assert_allclose(np.linalg.norm(nrm[key], axis=-1), np.sqrt(ss / (ss + 1e-6)),
                                   rtol=1e-13)
        # direction unchanged
        np.testing.assert_allclose(nrm[key] * np.sqrt(ss + 1e-6)[..., None], raw[key],
                                   rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(nrm["v"], raw["v"])


def test_split_resume_equals_whole():
    d = case([23])
    whole, pool_w = run(d)
    for t in (1, 2, 3, 4, 11, 22):
        a = dict(d, x=d["x"][:t], a=d["a"][:t], b=d["b"][:t], T=t,
                 cu=np.array([0, t], np.int32))
        out_a, pool_a = run(a)
        b = dict(d, x=d["x"][t:], a=d["a"][t:], b=d["b"][t:], T=d["T"] - t,
                 cu=np.array([0, d["T"] - t], np.int32), pool=pool_a)
        out_b, pool_b = run(b)
        for key in ("q", "k", "v", "g", "beta"):
            np.testing.assert_array_equal(np.concatenate([out_a[key], out_b[key]]), whole[key])
        np.testing.assert_array_equal(pool_b, pool_w)


def test_decode_batch_equals_single_tokens():
    d = case([1] * 6, slots=6)
    out, pool = run(d)
    for i in range(6):
        di = dict(d, x=d["x"][i:i + 1], a=d["a"][i:i + 1], b=d["b"][i:i + 1], T=1,
                  cu=np.array([0, 1], np.int32), pool=d["pool"][i:i + 1])
        oi, pi = run(di)
        for key in ("q", "k", "v", "g", "beta"):
            np.testing.assert_array_equal(out[key][i:i + 1], oi[key])
        np.testing.assert_array_equal(pool[i], pi[0])


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_thread_count_does_not_change_results(dtype):
    d = case([17, 4, 9], Hk=2, Dk=8, Dv=8)
    o1, p1 = run(d, norm=True, dtype=dtype, nthreads=1)
    o4, p4 = run(d, norm=True, dtype=dtype, nthreads=4)
    for key in o1:
        np.testing.assert_array_equal(o1[key], o4[key])
    np.testing.assert_array_equal(p1, p4)


def test_f32_matches_f64():
    d = case([40, 9], Hk=2, Dk=16, Dv=8)
    o32, p32 = run(d, norm=True, dtype=np.float32)
    o64, p64 = run(d, norm=True, dtype=np.float64)
    for key in o32:
        np.testing.assert_allclose(o32[key], o64[key], rtol=2e-5, atol=2e-6)
    np.testing.assert_allclose(p32, p64, rtol=1e-6)
