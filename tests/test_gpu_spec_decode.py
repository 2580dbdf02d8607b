"""GPU parity of gdn_spec_decode (speculative multi-token decode, [cpu_ops.cpp]
GdnSpecDecodeKernel) against the oracle, through the C ABI: every supported Dk,
bf16 and f32, negative initial slots and columns, empty requests, two chained
steps that resume from an accepted snapshot, the multi-token-prediction shape
at full size, and the device-side metadata checks.  The whole pool is compared:
snapshot slots against the oracle's, every other slot bit for bit."""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B

pytestmark = pytest.mark.gpu


def make(lens, num_cols, Hk, Hv, Dk, Dv, dtype, seed, slots=None):
    g0 = torch.Generator().manual_seed(seed)
    T, n = sum(lens), len(lens)
    slots = slots or n * num_cols + 3
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = (torch.randn(T, Hk, Dk, generator=g0) / np.sqrt(Dk)).to(dtype)
    k = (torch.randn(T, Hk, Dk, generator=g0) / np.sqrt(Dk)).to(dtype)
    v = torch.randn(T, Hv, Dv, generator=g0).to(dtype)
    g = -torch.rand(T, Hv, generator=g0) * 0.5
    beta = torch.rand(T, Hv, generator=g0) * 0.8 + 0.1
    pool = torch.randn(slots, Hv, Dv, Dk, generator=g0) * 0.1
    sidx = torch.randperm(slots, generator=g0)[:n * num_cols].reshape(n, num_cols).to(torch.int32)
    nat = torch.randint(1, num_cols + 1, (n,), generator=g0, dtype=torch.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, pool=pool, cu=cu, sidx=sidx, nat=nat)


def gpu_step(x, pool_d, dev, mirrors=True):
    T, Hv, Dv = x["v"].shape
    out = torch.full((T, Hv, Dv), 3.0, dtype=x["q"].dtype, device=dev)
    B.gdn_spec_decode(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), x["g"].to(dev),
                      x["beta"].to(dev), pool_d, x["cu"].to(dev), x["sidx"].to(dev),
                      x["nat"].to(dev), out,
                      cu_seqlens_host=x["cu"] if mirrors else None,
                      state_indices_host=x["sidx"] if mirrors else None,
                      num_accepted_host=x["nat"] if mirrors else None)
    return out


def oracle_step(x, ref_pool):
    Dk = x["q"].shape[2]
    return oracle.gdn_spec_decode(H.f32(x["q"]), H.f32(x["k"]), H.f32(x["v"]), x["g"].numpy(),
                                  x["beta"].numpy(), ref_pool, x["cu"].numpy(),
                                  x["sidx"].numpy(), x["nat"].numpy(), 1.0 / np.sqrt(Dk),
                                  dtype=np.float32)


def compare(x, out, pool_d, ref_out, ref_pool, before, what):
    tol = H.TOL_F32 if x["q"].dtype == torch.float32 else H.TOL_BF16
    H.check(out, ref_out, tol, what + " out")
    got = H.f32(pool_d)
    touched = sorted({int(s) for s in x["sidx"].flatten() if 0 <= s < before.shape[0]})
    untouched = [s for s in range(before.shape[0]) if s not in touched]
    assert np.array_equal(got[untouched], before[untouched]), what + ": untouched slots changed"
    if touched:
        H.assert_close(got[touched], ref_pool[touched], tol, what + " snapshots")


def run(lens, num_cols, Hk, Hv, Dk, Dv, dtype, dev, seed, edit=None, mirrors=True, slots=None):
    x = make(lens, num_cols, Hk, Hv, Dk, Dv, dtype, seed, slots)
    if edit is not None:
        edit(x)
    before = x["pool"].numpy().copy()
    pool_d = x["pool"].to(dev)
    out = gpu_step(x, pool_d, dev, mirrors)
    B.gdn_read_device_status()
    ref_pool = before.copy()
    ref_out = oracle_step(x, ref_pool)
    compare(x, out, pool_d, ref_out, ref_pool, before, "spec")
    return x, pool_d, ref_pool


@pytest.mark.parametrize("Dk", [16, 32, 64, 128, 256])
def test_spec_decode_all_dk(Dk, cuda_device):
    run([4, 1, 3, 2], 4, 2, 4, Dk, 64, torch.bfloat16, cuda_device, seed=Dk)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_spec_decode_rows_ragged_dv(dtype, cuda_device):
    # Dv = 80 leaves a partial row slice in every CTA
    run([3, 3, 1, 2, 3], 3, 1, 2, 128, 80, dtype, cuda_device, seed=2)


def test_spec_decode_null_slots_and_empty_requests(cuda_device):
    def edit(x):
        x["sidx"][0, x["nat"][0] - 1] = -1     # no initial state: outputs zero
        x["nat"][1] = 3
        x["sidx"][1, 1] = -7                   # request 1 skips one snapshot
    run([2, 3, 0, 4, 0], 4, 1, 2, 128, 64, torch.float32, cuda_device, seed=3, edit=edit)


def test_spec_decode_chained_steps_resume_from_accepted(cuda_device):
    """Step 1 drafts 4 tokens per request; step 2 resumes each request from
    the snapshot of its accepted prefix (the same slot row) -- the way a
    speculative decoder rolls back rejected drafts."""
    dev = cuda_device
    x1 = make([4] * 6, 4, 2, 4, 128, 128, torch.bfloat16, 7)
    x1["nat"][:] = 1
    before = x1["pool"].numpy().copy()
    pool_d = x1["pool"].to(dev)
    gpu_step(x1, pool_d, dev)
    ref_pool = before.copy()
    oracle_step(x1, ref_pool)
    x2 = make([4] * 6, 4, 2, 4, 128, 128, torch.bfloat16, 8)
    x2["sidx"] = x1["sidx"]
    x2["nat"] = torch.tensor([1, 2, 3, 4, 2, 1], dtype=torch.int32)
    mid = ref_pool.copy()
    out = gpu_step(x2, pool_d, dev)
    B.gdn_read_device_status()
    ref_out = oracle_step(x2, ref_pool)
    compare(x2, out, pool_d, ref_out, ref_pool, mid, "chained")


def test_spec_decode_mtp_full_size(cuda_device):
    """The multi-token-prediction decode the bench times: 128 requests x 4
    tokens, 16 key / 32 value heads of 128, bf16 activations, f32 pool."""
    run([4] * 128, 4, 16, 32, 128, 128, torch.bfloat16, cuda_device, seed=11)


def test_spec_decode_device_checks(cuda_device):
    """Without host mirrors the kernel checks the metadata itself: a
    num_accepted outside [1, num_cols] skips that request (outputs zero) and a
    request longer than its row is skipped; both raise the status word."""
    dev = cuda_device
    x = make([2, 2, 2], 3, 1, 2, 64, 64, torch.bfloat16, 5)
    x["nat"][1] = 4
    before = x["pool"].clone()
    pool_d = x["pool"].to(dev)
    out = gpu_step(x, pool_d, dev, mirrors=False)
    with pytest.raises(B.GdnError) as ei:
        B.gdn_read_device_status()
    assert ei.value.code == B.GDN_ERR_DEVICE_CHECK
    assert torch.all(out[2:4].float() == 0)
    assert torch.equal(pool_d.cpu()[x["sidx"][1].long()], before[x["sidx"][1].long()])
    # a request longer than its row (num_cols 3, request 0 has 4 tokens)
    y = make([4, 2], 3, 1, 2, 64, 64, torch.bfloat16, 6)
    pool_y = y["pool"].to(dev)
    gpu_step(y, pool_y, dev, mirrors=False)
    with pytest.raises(B.GdnError) as ei:
        B.gdn_read_device_status()
    assert ei.value.code == B.GDN_ERR_DEVICE_CHECK
    # the context is still usable
    run([1, 2], 2, 1, 2, 64, 64, torch.bfloat16, dev, seed=8)
