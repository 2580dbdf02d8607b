"""Pins of the oracle's recurrence (O2 sequential, O3 decode, O4 chunked).

Follows [cpu.rs] (ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs)
recurrent_gated_delta_rule_varlen_f32 and [cpu_ops.cpp] (vllm.cpp,
src/vt/cpu/cpu_ops.cpp) GdnHeadTokenStep / GdnDecodeKernel.  Pins:
  - matrix (Householder) form, brute force in numpy:
        S_t = e^g S_{t-1} (I - beta k k^T) + beta v k^T,  o_t = S_t (scale q)
    which is algebraically the pages' update but a different expression;
  - g = 0, beta = 0: S constant, o = S (scale q) exactly;
  - g = 0, beta = 1, orthonormal keys: exact delta-rule overwrite S k_s = v_s;
  - one token from zero state: S = beta v k^T, o = beta scale (k.q) v;
  - beta = 0: S_T = exp(sum g) S_0;
  - GQA: value head h reads key head h / (Hv/Hk) (duplicated key heads give the
    same result as Hk = Hv);
  - the chunked WY/UT form (derived, f64) equals the sequential form to 1e-12
    for T in {1, 63, 64, 65, 130}, chunk in {4, 16, 64}, varlen, carried state;
  - split/resume with the carried state == one run; decode x T == prefill;
  - -1 slot: zero output, pool untouched; has_initial_state = 0: zero start.
"""
import numpy as np
import pytest

import oracle


def rand_case(seqlens, Hk=1, Hv=2, Dk=4, Dv=3, seed=0, gscale=0.3, slots=None, unit_keys=True):
    rng = np.random.default_rng(seed)
    T = int(sum(seqlens))
    q = rng.normal(size=(T, Hk, Dk))
    k = rng.normal(size=(T, Hk, Dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(T, Hv, Dv))
    g = -np.abs(rng.normal(size=(T, Hv))) * gscale
    beta = rng.uniform(0.05, 0.95, size=(T, Hv))
    slots = slots or len(seqlens)
    pool = rng.normal(size=(slots, Hv, Dv, Dk)) * 0.5
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, pool=pool, cu=cu)


def seq(d, scale=0.7, dtype=np.float64, **kw):
    pool = d["pool"].astype(dtype).copy()
    out = oracle.gdn_varlen(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["cu"], scale,
                            dtype=dtype, **kw)
    return out, pool


def householder(q, k, v, g, beta, S0, scale):
    """Matrix form for one (sequence, value head): lists of o_t and S_T."""
    S = S0.copy()
    I = np.eye(S.shape[1])
    outs = []
    for t in range(q.shape[0]):
        S = np.exp(g[t]) * S @ (I - beta[t] * np.outer(k[t], k[t])) + beta[t] * np.outer(v[t], k[t])
        outs.append(S @ (scale * q[t]))
    return np.array(outs), S


def test_matches_householder_form():
    d = rand_case([9, 5, 14], Hk=2, Hv=4, Dk=6, Dv=5, seed=1)
    out, pool = seq(d, scale=0.4)
    ratio = 2
    for s in range(3):
        lo, hi = d["cu"][s], d["cu"][s + 1]
        for h in range(4):
            hk = h // ratio
            o, S = householder(d["q"][lo:hi, hk], d["k"][lo:hi, hk], d["v"][lo:hi, h],
                               d["g"][lo:hi, h], d["beta"][lo:hi, h], d["pool"][s, h], 0.4)
            np.testing.assert_allclose(out[lo:hi, h], o, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(pool[s, h], S, rtol=1e-12, atol=1e-13)


def test_qk_l2norm_in_loop_equals_prenormalised():
    d = rand_case([11], Hk=1, Hv=2, Dk=5, Dv=3, seed=2, unit_keys=False)
    out_n, pool_n = seq(d, use_qk_l2norm=True)
    dd = dict(d)
    dd["q"] = d["q"] / np.sqrt((d["q"] ** 2).sum(-1, keepdims=True) + 1e-6)
    dd["k"] = d["k"] / np.sqrt((d["k"] ** 2).sum(-1, keepdims=True) + 1e-6)
    out_p, pool_p = seq(dd)
    np.testing.assert_allclose(out_n, out_p, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(pool_n, pool_p, rtol=1e-12, atol=1e-13)


def test_constant_state_when_g_and_beta_zero():
    d = rand_case([7], Hv=2)
    d["g"][:] = 0.0
    d["beta"][:] = 0.0
    out, pool = seq(d, scale=0.9)
    np.testing.assert_array_equal(pool, d["pool"])
    for h in range(2):
        np.testing.assert_allclose(out[:, h], (0.9 * d["q"][:, 0]) @ d["pool"][0, h].T,
                                   rtol=1e-13)


def test_exact_overwrite_with_orthonormal_keys():
    Dk = Dv = 8
    rng = np.random.default_rng(3)
    Qm, _ = np.linalg.qr(rng.normal(size=(Dk, Dk)))
    d = rand_case([Dk], Hk=1, Hv=1, Dk=Dk, Dv=Dv, seed=4)
    d["k"][:, 0] = Qm.T  # rows are orthonormal
    d["g"][:] = 0.0
    d["beta"][:] = 1.0
    out, pool = seq(d)
    S = pool[0, 0]
    # every stored association is recalled exactly: S k_s = v_s
    np.testing.assert_allclose(S @ d["k"][:, 0].T, d["v"][:, 0].T, atol=1e-12)


def test_one_token_from_zero_state():
    d = rand_case([1], Hk=1, Hv=1, Dk=5, Dv=4, seed=5)
    d["pool"][:] = 0.0
    out, pool = seq(d, scale=0.3)
    b, k, q, v = d["beta"][0, 0], d["k"][0, 0], d["q"][0, 0], d["v"][0, 0]
    np.testing.assert_allclose(pool[0, 0], b * np.outer(v, k), rtol=1e-14)
    np.testing.assert_allclose(out[0, 0], b * 0.3 * (k @ q) * v, rtol=1e-13)


def test_decay_only():
    d = rand_case([6], Hv=2, seed=6)
    d["beta"][:] = 0.0
    out, pool = seq(d)
    for h in range(2):
        np.testing.assert_allclose(pool[0, h], np.exp(d["g"][:, h].sum()) * d["pool"][0, h],
                                   rtol=1e-13)


def test_gqa_mapping():
    # Hk = 2, Hv = 4: heads 0,1 read key head 0; heads 2,3 read key head 1
    d = rand_case([8], Hk=2, Hv=4, seed=7)
    out, pool = seq(d)
    dd = dict(d)
    dd["q"] = np.repeat(d["q"], 2, axis=1)  # [T, 4, Dk] with q[:, h] = q[:, h // 2]
    dd["k"] = np.repeat(d["k"], 2, axis=1)
    out2, pool2 = seq(dd)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(pool, pool2)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
@pytest.mark.parametrize("chunk", [4, 16, 64])
def test_chunked_equals_sequential(T, chunk):
    d = rand_case([T], Hk=1, Hv=2, Dk=4, Dv=8, seed=T * 7 + chunk, gscale=0.5)
    ref, pool_ref = seq(d, scale=0.6)
    pool = d["pool"].copy()
    out = oracle.gdn_chunked_f64(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["cu"], 0.6,
                                 chunk)
    rms = np.sqrt((ref ** 2).mean())
    assert np.abs(out - ref).max() <= 1e-12 * max(rms, 1.0)
    assert np.abs(pool - pool_ref).max() <= 1e-12 * max(np.sqrt((pool_ref ** 2).mean()), 1.0)


def test_chunked_varlen_mixed_metadata():
    d = rand_case([5, 70, 1, 33], Hk=2, Hv=4, Dk=8, Dv=4, seed=11, slots=6, gscale=0.2,
                  unit_keys=False)
    sidx = np.array([5, 0, -1, 2], np.int32)
    hinit = np.array([1, 0, 1, 1], np.uint8)
    for norm in (False, True):
        ref, pool_ref = seq(d, state_indices=sidx, has_initial_state=hinit, use_qk_l2norm=norm)
        pool = d["pool"].copy()
        out = oracle.gdn_chunked_f64(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["cu"],
                                     0.7, 16, state_indices=sidx, has_initial_state=hinit,
                                     use_qk_l2norm=norm)
        np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(pool, pool_ref, rtol=1e-11, atol=1e-12)


def test_padding_and_zero_start():
    d = rand_case([4, 3, 5], Hv=2, seed=12, slots=5)
    sidx = np.array([3, -1, 0], np.int32)
    hinit = np.array([0, 1, 1], np.uint8)
    out, pool = seq(d, state_indices=sidx, has_initial_state=hinit)
    np.testing.assert_array_equal(out[4:7], 0.0)          # padded sequence 1
    for untouched in (1, 2, 4):
        np.testing.assert_array_equal(pool[untouched], d["pool"][untouched])
    # sequence 0 started from zero in slot 3
    dz = dict(d)
    p = d["pool"].copy()
    p[3] = 0.0
    dz["pool"] = p
    out_z, pool_z = seq(dz, state_indices=sidx)
    np.testing.assert_array_equal(out[0:4], out_z[0:4])
    np.testing.assert_array_equal(pool[3], pool_z[3])


def test_split_resume_equals_whole():
    d = rand_case([50], Hv=2, seed=13)
    whole, pool_w = seq(d)
    for t in (1, 17, 49):
        a = dict(d, q=d["q"][:t], k=d["k"][:t], v=d["v"][:t], g=d["g"][:t], beta=d["beta"][:t],
                 cu=np.array([0, t], np.int32))
        oa, pa = seq(a)
        b = dict(d, q=d["q"][t:], k=d["k"][t:], v=d["v"][t:], g=d["g"][t:], beta=d["beta"][t:],
                 cu=np.array([0, 50 - t], np.int32), pool=pa)
        ob, pb = seq(b)
        np.testing.assert_array_equal(np.concatenate([oa, ob]), whole)
        np.testing.assert_array_equal(pb, pool_w)


def test_decode_repeated_equals_prefill():
    d = rand_case([12], Hk=2, Hv=4, seed=14)
    whole, pool_w = seq(d)
    pool = d["pool"].copy()
    outs = []
    for t in range(12):
        outs.append(oracle.gdn_decode(d["q"][t:t + 1], d["k"][t:t + 1], d["v"][t:t + 1],
                                      d["g"][t:t + 1], d["beta"][t:t + 1], pool, 0.7,
                                      dtype=np.float64))
    np.testing.assert_array_equal(np.concatenate(outs), whole)
    np.testing.assert_array_equal(pool, pool_w)


def test_decode_negative_index():
    d = rand_case([1, 1, 1], Hv=2, seed=15, slots=4)
    pool = d["pool"].copy()
    out = oracle.gdn_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, 0.5,
                            state_indices=np.array([2, -1, 0], np.int32), dtype=np.float64)
    np.testing.assert_array_equal(out[1], 0.0)
    np.testing.assert_array_equal(pool[1], d["pool"][1])
    np.testing.assert_array_equal(pool[3], d["pool"][3])


def test_items_subset_matches_full():
    d = rand_case([9, 4], Hk=1, Hv=3, seed=16)
    full, pool_full = seq(d)
    pool = d["pool"].copy()
    out = oracle.gdn_varlen(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["cu"], 0.7,
                            items=np.array([4, 0], np.int32), dtype=np.float64)
    np.testing.assert_array_equal(out[9:, 1], full[9:, 1])  # item 4 = seq 1, head 1
    np.testing.assert_array_equal(out[:9, 0], full[:9, 0])  # item 0 = seq 0, head 0
    np.testing.assert_array_equal(pool[1, 1], pool_full[1, 1])


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_thread_count_does_not_change_results(dtype):
    d = rand_case([30, 7, 19], Hk=2, Hv=4, Dk=8, Dv=8, seed=17)
    o1, p1 = seq(d, dtype=dtype, nthreads=1)
    o8, p8 = seq(d, dtype=dtype, nthreads=8)
    np.testing.assert_array_equal(o1, o8)
    np.testing.assert_array_equal(p1, p8)


def test_f32_close_to_f64():
    d = rand_case([40], Hk=2, Hv=4, Dk=16, Dv=16, seed=18)
    o32, p32 = seq(d, dtype=np.float32)
    o64, p64 = seq(d, dtype=np.float64)
    assert np.abs(o32 - o64).max() <= 1e-5 * np.sqrt((o64 ** 2).mean())
    assert np.abs(p32 - p64).max() <= 1e-5 * np.sqrt((p64 ** 2).mean())
