"""Device-side checks: with no host mirror, a state index outside [-1, slots)
is caught by the kernel, which skips the sequence and raises the device status
word (read back as GDN_ERR_DEVICE_CHECK); nothing is accessed out of bounds
and the context stays usable.  Also: every slot the call does not own is left
bit-identical, and a later good call succeeds.  A bounded wait that runs out
is reported as GDN_ERR_TIMEOUT the same way."""
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


@pytest.mark.parametrize("algo", [B.GDN_PREFILL_RECURRENT, B.GDN_PREFILL_CHUNKED,
                                  B.GDN_PREFILL_FUSED])
def test_bad_cu_seqlens_is_reported(algo, cuda_device):
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
    nbytes = B.gdn_prefill_workspace_bytes(T, N, Hv, D, D, B.GDN_DTYPE_BF16, algo)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev) if nbytes else None
    B.gdn_prefill_varlen(q, k, v, g, beta, pool, cu, out, algo=algo, workspace=ws)
    with pytest.raises(B.GdnError) as ei:
        B.gdn_read_device_status()
    assert ei.value.code == B.GDN_ERR_DEVICE_CHECK


def test_wait_timeout_is_reported_and_the_context_stays_usable(cuda_device):
    """A bounded device wait that runs out (an mbarrier nothing arrives on,
    nothing else in flight) records GDN_ERR_TIMEOUT in the status word; reading
    it clears it, and the next calls run normally."""
    dev = cuda_device
    B.gdn_read_device_status()  # a clean word to start from
    B.gdn_check_wait_timeout(2_000_000)  # about a millisecond of SM clock
    with pytest.raises(B.GdnError) as ei:
        B.gdn_read_device_status()
    assert ei.value.code == B.GDN_ERR_TIMEOUT
    B.gdn_read_device_status()  # cleared
    with pytest.raises(B.GdnError) as ei:
        B.gdn_check_wait_timeout(0)
    assert ei.value.code == B.GDN_ERR_INVALID_ARGUMENT
    # a good call afterwards: one decode, checked against the row update by hand
    q = torch.zeros(1, 1, 128, device=dev, dtype=torch.bfloat16)
    q[0, 0, 0] = 1.0
    k = q.clone()
    v = torch.full((1, 1, 128), 2.0, device=dev, dtype=torch.bfloat16)
    g = torch.zeros(1, 1, device=dev)
    beta = torch.ones(1, 1, device=dev)
    pool = torch.zeros(1, 1, 128, 128, device=dev)
    out = torch.empty(1, 1, 128, dtype=torch.bfloat16, device=dev)
    B.gdn_decode(q, k, v, g, beta, pool, out, scale=1.0)
    B.gdn_read_device_status()
    # S = beta v k^T = 2 e_0^T per row; o = S q = 2
    assert torch.all(out.float() == 2.0)
    assert torch.all(pool[0, 0, :, 0] == 2.0) and pool[0, 0, :, 1:].abs().max() == 0
