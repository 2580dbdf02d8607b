"""GPU parity of gdn_spec_prepare (the prepare step of a speculative decode:
[cpu_ops.cpp] CausalConv1dSpecUpdateKernel, then split, norm and gates)
against the oracle, through the C ABI: the multi-token-prediction shape, ragged
and empty requests, a negative conv row, conv widths 2..8 with rows of up to
14 entries, warps that hold both key and value channels, two chained steps,
a whole speculative step (prepare then decode), and the device-side checks.
The conv rows hold raw inputs only, so the pool must match bit for bit."""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B

pytestmark = pytest.mark.gpu


def make(lens, max_q, Hk, Hv, Dk, Dv, K, dtype, seed, slots=None):
    g0 = torch.Generator().manual_seed(seed)
    T, n = sum(lens), len(lens)
    C = 2 * Hk * Dk + Hv * Dv
    width = (K - 1) + (max_q - 1)
    slots = slots or n + 3
    return dict(
        x=torch.randn(T, C, generator=g0).to(dtype),
        w=torch.randn(C, K, generator=g0) * 0.4,
        a=torch.randn(T, Hv, generator=g0).to(dtype),
        b=torch.randn(T, Hv, generator=g0).to(dtype),
        A_log=torch.randn(Hv, generator=g0) * 0.3,
        dt_bias=torch.randn(Hv, generator=g0) * 0.3,
        pool=torch.randn(slots, C, width, generator=g0).to(dtype).float(),
        cu=torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32),
        idx=torch.randperm(slots, generator=g0)[:n].to(torch.int32),
        nat=torch.randint(1, max_q + 1, (n,), generator=g0, dtype=torch.int32),
        dims=(Hk, Hv, Dk, Dv, K), dtype=dtype)


def gpu_step(d, pool_d, dev, mirrors=True, norm=True):
    Hk, Hv, Dk, Dv, K = d["dims"]
    T = d["x"].shape[0]
    q = torch.empty(T, Hk, Dk, dtype=d["dtype"], device=dev)
    k = torch.empty_like(q)
    v = torch.empty(T, Hv, Dv, dtype=d["dtype"], device=dev)
    g = torch.empty(T, Hv, device=dev)
    beta = torch.empty_like(g)
    B.gdn_spec_prepare(d["x"].to(dev), d["w"].to(dev), d["a"].to(dev), d["b"].to(dev),
                       d["A_log"].to(dev), d["dt_bias"].to(dev), d["cu"].to(dev), pool_d,
                       d["idx"].to(dev), d["nat"].to(dev), q, k, v, g, beta, Hk=Hk, Hv=Hv,
                       Dk=Dk, Dv=Dv, K=K, cu_seqlens_host=d["cu"] if mirrors else None,
                       conv_indices_host=d["idx"] if mirrors else None,
                       num_accepted_host=d["nat"] if mirrors else None, apply_qk_l2norm=norm)
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def oracle_step(d, ref_pool, norm=True):
    Hk, Hv, Dk, Dv, K = d["dims"]
    return oracle.spec_prepare(H.f32(d["x"]), d["w"].numpy(), ref_pool, H.f32(d["a"]),
                               H.f32(d["b"]), d["A_log"].numpy(), d["dt_bias"].numpy(),
                               d["cu"].numpy(), d["idx"].numpy(), d["nat"].numpy(), Hk, Hv, Dk,
                               Dv, K, apply_qk_l2norm=norm, dtype=np.float32)


def compare(d, got, ref, pool_d, ref_pool):
    tol = H.TOL_F32 if d["dtype"] == torch.float32 else H.TOL_BF16
    T = d["x"].shape[0]
    for name in ("q", "k", "v"):
        H.check(got[name], ref[name], tol, "spec prepare " + name)
    for name in ("g", "beta"):
        H.assert_close(H.f32(got[name]), ref[name].reshape(T, -1), H.TOL_F32, name)
    np.testing.assert_array_equal(H.f32(pool_d), ref_pool)


def run(lens, max_q, Hk, Hv, Dk, Dv, K, dtype, dev, seed, edit=None, norm=True):
    d = make(lens, max_q, Hk, Hv, Dk, Dv, K, dtype, seed)
    if edit is not None:
        edit(d)
    ref_pool = d["pool"].numpy().copy()
    pool_d = d["pool"].to(dev)
    got = gpu_step(d, pool_d, dev, norm=norm)
    B.gdn_read_device_status()
    ref = oracle_step(d, ref_pool, norm=norm)
    compare(d, got, ref, pool_d, ref_pool)


def test_spec_prepare_mtp_full_size(cuda_device):
    """128 requests x 4 drafts, 16 key / 32 value heads of 128, K = 4."""
    run([4] * 128, 4, 16, 32, 128, 128, 4, torch.bfloat16, cuda_device, seed=1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_spec_prepare_ragged_null_row_mixed_warps(dtype, cuda_device):
    # 2*Hk*Dk = 128 channels: the first warp holds key and value lanes
    def edit(d):
        d["idx"][3] = -1
    run([3, 0, 1, 4, 2, 4], 4, 2, 4, 32, 16, 4, dtype, cuda_device, seed=2, edit=edit)


@pytest.mark.parametrize("K,max_q", [(2, 1), (2, 8), (4, 2), (8, 8), (6, 5)])
def test_spec_prepare_conv_widths(K, max_q, cuda_device):
    # (8, 8): a row of 14 entries, 57 KB of staging (above the 48 KB default)
    lens = [max_q, max(1, max_q - 1), max_q, 1]
    run(lens, max_q, 1, 2, 64, 64, K, torch.bfloat16, cuda_device, seed=10 * K + max_q)


def test_spec_prepare_without_norm(cuda_device):
    run([2, 3, 3], 3, 2, 4, 64, 32, 4, torch.float32, cuda_device, seed=5, norm=False)


def test_spec_prepare_chained_steps(cuda_device):
    """Step 2 reads the rows step 1 wrote, at its own accepted offsets."""
    dev = cuda_device
    d1 = make([4] * 8, 4, 2, 4, 128, 64, 4, torch.bfloat16, 6)
    ref_pool = d1["pool"].numpy().copy()
    pool_d = d1["pool"].to(dev)
    gpu_step(d1, pool_d, dev)
    oracle_step(d1, ref_pool)
    d2 = make([4] * 8, 4, 2, 4, 128, 64, 4, torch.bfloat16, 7)
    d2["idx"], d2["w"] = d1["idx"], d1["w"]
    got = gpu_step(d2, pool_d, dev)
    B.gdn_read_device_status()
    ref = oracle_step(d2, ref_pool)
    compare(d2, got, ref, pool_d, ref_pool)


def test_spec_step_prepare_then_decode(cuda_device):
    """A whole speculative step through the ABI: gdn_spec_prepare feeds
    gdn_spec_decode; the oracle chain rounds q, k, v to bf16 between its
    steps, as the GPU path stores them."""
    dev = cuda_device
    n, max_q, Hk, Hv, D = 16, 4, 4, 8, 128
    d = make([max_q] * n, max_q, Hk, Hv, D, D, 4, torch.bfloat16, 8)
    g0 = torch.Generator().manual_seed(9)
    slots = n * max_q + 2
    spool = torch.randn(slots, Hv, D, D, generator=g0) * 0.05
    sidx = torch.randperm(slots, generator=g0)[:n * max_q].reshape(n, max_q).to(torch.int32)
    ref_conv = d["pool"].numpy().copy()
    conv_d = d["pool"].to(dev)
    prep = gpu_step(d, conv_d, dev)
    spool_d = spool.to(dev)
    out = torch.empty(n * max_q, Hv, D, dtype=torch.bfloat16, device=dev)
    B.gdn_spec_decode(prep["q"], prep["k"], prep["v"], prep["g"], prep["beta"], spool_d,
                      d["cu"].to(dev), sidx.to(dev), d["nat"].to(dev), out,
                      cu_seqlens_host=d["cu"], state_indices_host=sidx,
                      num_accepted_host=d["nat"])
    B.gdn_read_device_status()
    ref = oracle_step(d, ref_conv)
    ref_spool = spool.numpy().copy()
    ref_out = oracle.gdn_spec_decode(H.bf16_round(ref["q"]), H.bf16_round(ref["k"]),
                                     H.bf16_round(ref["v"]), ref["g"], ref["beta"], ref_spool,
                                     d["cu"].numpy(), sidx.numpy(), d["nat"].numpy(),
                                     1.0 / np.sqrt(D), dtype=np.float32)
    H.check(out, ref_out, H.TOL_BF16, "spec step out")
    touched = sorted({int(s) for s in sidx.flatten()})
    H.assert_close(H.f32(spool_d)[touched], ref_spool[touched], H.TOL_BF16, "spec step states")


def test_spec_prepare_device_checks(cuda_device):
    """Without host mirrors: a num_accepted outside [1, max_q] raises the
    status word, the request's outputs come from a zero window and its row is
    left alone; a request longer than max_q is skipped."""
    dev = cuda_device
    d = make([2, 3, 1], 3, 1, 2, 64, 64, 4, torch.bfloat16, 11)
    d["nat"][1] = 4
    ref_pool = d["pool"].numpy().copy()
    pool_d = d["pool"].to(dev)
    got = gpu_step(d, pool_d, dev, mirrors=False)
    with pytest.raises(B.GdnError) as ei:
        B.gdn_read_device_status()
    assert ei.value.code == B.GDN_ERR_DEVICE_CHECK
    d_ref = dict(d)
    d_ref["idx"] = d["idx"].clone()
    d_ref["idx"][1] = -1                     # what the kernel falls back to
    d_ref["nat"] = d["nat"].clone()
    d_ref["nat"][1] = 1
    ref = oracle_step(d_ref, ref_pool)
    compare(d, got, ref, pool_d, ref_pool)
    e = make([4, 2], 3, 1, 2, 64, 64, 4, torch.bfloat16, 12)
    gpu_step(e, e["pool"].to(dev), dev, mirrors=False)
    with pytest.raises(B.GdnError) as ei:
        B.gdn_read_device_status()
    assert ei.value.code == B.GDN_ERR_DEVICE_CHECK
    run([1, 2], 2, 1, 2, 64, 64, 4, torch.bfloat16, dev, seed=13)
