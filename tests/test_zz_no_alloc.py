"""gdn_prefill_varlen_noalloc: the chunked prefill for callers that cannot
allocate device memory (a plug-in whose host runtime owns all device memory and
offers no allocator, or a serving loop that must never call cudaMalloc).  It
takes the same arguments as gdn_prefill_varlen but uses the library's fixed
64 MiB device scratch instead of a caller workspace.

Checked through the C ABI: the allocating entry point's result is first
checked against the oracle within the parity tolerance; then two no-alloc calls
in a row (the second finds the first call's leftovers in the shared scratch)
must each reproduce it bit for bit, since they run the same kernels on the same
inputs.  Sizes beyond the scratch are rejected before anything is launched.  This file is collected last so that
a run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process (the first call sets up the device
address of the scratch)."""
import ctypes

import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B
from gated_delta_rule_44_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc():
    L = B.lib()
    fn = L.gdn_prefill_varlen_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(B.gdn_prefill_args), ctypes.c_void_p]
    return fn


def _args(q, k, v, g, beta, state, cu, sidx, hinit, out, algo=B.GDN_PREFILL_CHUNKED):
    T, Hk, Dk = q.shape
    _, Hv, Dv = v.shape
    return B.gdn_prefill_args(
        T=T, N=cu.numel() - 1, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act_dtype=B.GDN_DTYPE_BF16,
        use_qk_l2norm=0, scale=-1.0, algo=algo, q=q.data_ptr(), q_len=q.numel(),
        k=k.data_ptr(), k_len=k.numel(), v=v.data_ptr(), v_len=v.numel(), g=g.data_ptr(),
        g_len=g.numel(), beta=beta.data_ptr(), beta_len=beta.numel(), state=state.data_ptr(),
        state_slots=state.shape[0], state_len=state.numel(), cu_seqlens=cu.data_ptr(),
        state_indices=sidx.data_ptr(), has_initial_state=hinit.data_ptr(), cu_seqlens_host=None,
        state_indices_host=None, out=out.data_ptr(), out_len=out.numel(), workspace=None,
        workspace_bytes=0)


def test_noalloc_matches_allocating_entry_point(cuda_device):
    dev = cuda_device
    w = W.make_workload("noalloc", 900, [70, 1, 200, 129], 4, 8, 128, 128, slots=6,
                        weak_decay=True, state_std=0.3)
    need = B.gdn_prefill_workspace_bytes(w.T, w.N, w.Hv, w.Dk, w.Dv, B.GDN_DTYPE_BF16,
                                         B.GDN_PREFILL_CHUNKED)
    assert 0 < need <= 64 << 20
    prep, _ = H.oracle_prepare(w)
    q, k, v = (torch.from_numpy(prep[x]).to(torch.bfloat16).to(dev) for x in ("q", "k", "v"))
    g = torch.from_numpy(prep["g"]).to(dev)
    beta = torch.from_numpy(prep["beta"]).to(dev)
    cu = w.cu_seqlens.to(dev)
    sidx = w.state_indices.to(dev)
    hinit = w.has_initial_state.to(dev)

    # reference: the allocating entry point with a torch-allocated workspace
    state_ref = w.state_pool.to(dev)
    out_ref = torch.empty((w.T, w.Hv, w.Dv), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    B.gdn_prefill_varlen(q, k, v, g, beta, state_ref, cu, out_ref, state_indices=sidx,
                         has_initial_state=hinit, algo=B.GDN_PREFILL_CHUNKED, workspace=ws)
    torch.cuda.synchronize()
    B.gdn_read_device_status()
    # the reference itself against the oracle's recurrence (O2)
    pool = w.state_pool.numpy().copy()
    ref_o = oracle.gdn_varlen(H.f32(q), H.f32(k), H.f32(v), prep["g"], prep["beta"], pool,
                              w.cu_seqlens.numpy(), 1.0 / np.sqrt(w.Dk),
                              state_indices=w.state_indices.numpy(),
                              has_initial_state=w.has_initial_state.numpy(), dtype=np.float32)
    H.assert_close(H.f32(out_ref), ref_o, H.TOL_BF16, "allocating out", stored_bf16=True)
    H.assert_close(H.f32(state_ref), pool, H.TOL_BF16, "allocating state")

    fn = _noalloc()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        state = w.state_pool.to(dev)
        out = torch.full((w.T, w.Hv, w.Dv), float("nan"), dtype=torch.bfloat16, device=dev)
        a = _args(q, k, v, g, beta, state, cu, sidx, hinit, out)
        rc = fn(ctypes.byref(a), stream)
        assert rc == B.GDN_OK, B.lib().gdn_last_error_message().decode()
        B.gdn_read_device_status()
        assert torch.equal(out, out_ref), f"out (call {call}) differs from the allocating call"
        assert torch.equal(state, state_ref), f"state (call {call}) differs"


def test_noalloc_fused_spread(cuda_device):
    """The fused form with more chains than SMs takes its schedule's workspace
    from the scratch too: bit for bit the allocating call with a workspace,
    and the one-CTA-per-chain call without one."""
    dev = cuda_device
    w = W.make_workload("noalloc", 901, [int(x) for x in np.random.default_rng(10).integers(1, 260, 44)],
                        2, 4, 128, 128, weak_decay=True, state_std=0.3)
    assert w.N * w.Hv > torch.cuda.get_device_properties(dev).multi_processor_count
    need = B.gdn_prefill_workspace_bytes(w.T, w.N, w.Hv, w.Dk, w.Dv, B.GDN_DTYPE_BF16,
                                         B.GDN_PREFILL_FUSED)
    assert 0 < need <= 64 << 20
    prep, _ = H.oracle_prepare(w)
    q, k, v = (torch.from_numpy(prep[x]).to(torch.bfloat16).to(dev) for x in ("q", "k", "v"))
    g = torch.from_numpy(prep["g"]).to(dev)
    beta = torch.from_numpy(prep["beta"]).to(dev)
    cu, sidx, hinit = (x.to(dev) for x in (w.cu_seqlens, w.state_indices, w.has_initial_state))
    results = []
    for ws in (torch.empty(need, dtype=torch.uint8, device=dev), None):
        state = w.state_pool.to(dev)
        out = torch.empty((w.T, w.Hv, w.Dv), dtype=torch.bfloat16, device=dev)
        B.gdn_prefill_varlen(q, k, v, g, beta, state, cu, out, state_indices=sidx,
                             has_initial_state=hinit, algo=B.GDN_PREFILL_FUSED, workspace=ws)
        B.gdn_read_device_status()
        results.append((out, state))
    state = w.state_pool.to(dev)
    out = torch.full((w.T, w.Hv, w.Dv), float("nan"), dtype=torch.bfloat16, device=dev)
    a = _args(q, k, v, g, beta, state, cu, sidx, hinit, out, algo=B.GDN_PREFILL_FUSED)
    n0 = B.gdn_launch_count()
    rc = _noalloc()(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert rc == B.GDN_OK, B.lib().gdn_last_error_message().decode()
    assert B.gdn_launch_count() - n0 == 2  # the schedule kernel, then the fused kernel
    B.gdn_read_device_status()
    for ref_out, ref_state in results:
        assert torch.equal(out, ref_out)
        assert torch.equal(state, ref_state)


def test_noalloc_rejects_sizes_beyond_the_scratch(cuda_device):
    dev = cuda_device
    T, Hk, Hv, D = 20000, 1, 64, 128   # (20000/64 + 1) * 64 blobs: far beyond 64 MiB
    q = torch.zeros((T, Hk, D), dtype=torch.bfloat16, device=dev)
    v = torch.zeros((T, Hv, D), dtype=torch.bfloat16, device=dev)
    g = torch.zeros((T, Hv), device=dev)
    state = torch.zeros((1, Hv, D, D), device=dev)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    sidx = torch.zeros(1, dtype=torch.int32, device=dev)
    hinit = torch.ones(1, dtype=torch.uint8, device=dev)
    out = torch.zeros((T, Hv, D), dtype=torch.bfloat16, device=dev)
    launches = B.gdn_launch_count()
    a = _args(q, q, v, g, g, state, cu, sidx, hinit, out)
    rc = _noalloc()(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert rc == B.GDN_ERR_INVALID_ARGUMENT
    assert "workspace needs" in B.lib().gdn_last_error_message().decode()
    assert B.gdn_launch_count() == launches
