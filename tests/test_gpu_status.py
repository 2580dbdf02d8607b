"""Device-side checks: with no host mirror, a state index outside [-1, slots)
is caught by the kernel, which skips the sequence and raises the device status
word (read back as GDN_ERR_DEVICE_CHECK); nothing is accessed out of bounds
and the context stays usable.  Also: every slot the call does not own is left
bit-identical, and a later good call succeeds."""
import numpy as np
import pytest
import torch

from gated_delta_rule_44_gb300 import binding as B

pytestmark = pytest.mark.gpu


def test_bad_index_is_reported_not_faulted(cuda_device):
    dev = cuda_device
    Bn, Hk, Hv, D = 4, 1, 2, 128
    q = torch.randn(Bn, Hk, D, device=dev).to(torch.bfloat16)
    k = torch.randn(Bn, Hk, D, device=dev).to(torch.bfloat16)
    v = torch.randn(Bn, Hv, D, device=dev).to(torch.bfloat16)
    g = -torch.rand(Bn, Hv, device=dev)
    beta = torch.rand(Bn, Hv, device=dev)
    pool = torch.randn(3, Hv, D, D, device=dev)
    before = pool.clone()
    out = torch.empty(Bn, Hv, D, dtype=torch.bfloat16, device=dev)
    idx = torch.tensor([0, 7, -1, -5], dtype=torch.int32, device=dev)
    B.gdn_decode(q, k, v, g, beta, pool, out, state_indices=idx)
    with pytest.raises(B.GdnError) as ei:
        B.gdn_read_device_status()
    assert ei.value.code == B.GDN_ERR_DEVICE_CHECK
    assert torch.equal(pool[1:], before[1:])
    assert torch.all(out[1:].float() == 0)
    # the context is still usable and the status word was cleared
    B.gdn_decode(q, k, v, g, beta, pool, out, state_indices=torch.tensor(
        [0, 1, 2, -1], dtype=torch.int32, device=dev))
    B.gdn_read_device_status()


def test_bad_cu_seqlens_is_reported(cuda_device):
    dev = cuda_device
    T, N, Hk, Hv, D = 8, 2, 1, 2, 128
    q = torch.randn(T, Hk, D, device=dev).to(torch.bfloat16)
    k = torch.randn(T, Hk, D, device=dev).to(torch.bfloat16)
    v = torch.randn(T, Hv, D, device=dev).to(torch.bfloat16)
    g = -torch.rand(T, Hv, device=dev)
    beta = torch.rand(T, Hv, device=dev)
    pool = torch.randn(N, Hv, D, D, device=dev)
    out = torch.empty(T, Hv, D, dtype=torch.bfloat16, device=dev)
    cu = torch.tensor([0, 9, 8], dtype=torch.int32, device=dev)  # decreasing, out of range
    B.gdn_prefill_varlen(q, k, v, g, beta, pool, cu, out, algo=B.GDN_PREFILL_RECURRENT)
    with pytest.raises(B.GdnError) as ei:
        B.gdn_read_device_status()
    assert ei.value.code == B.GDN_ERR_DEVICE_CHECK
