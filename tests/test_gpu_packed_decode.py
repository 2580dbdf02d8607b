"""GPU parity of gdn_packed_decode (decode in one launch from the packed
projections: [cpu_ops.cpp] GdnPackedDecodeKernel with the conv update of
CausalConv1dUpdateKernel folded in; packed layouts of [cpu.rs]
linear_attention_prepare_varlen_packed_qkvz_ba_f32) against the oracle's
prepare (O1) followed by its decode (O3), computed in f64, through the C ABI.
Between the two steps the reference rounds beta through b's storage type (bf16,
nearest even) where the page's kernel does so, "exactly at the upstream
store/load boundary"; nothing else is rounded in between.  Covers the decode_b256 shape, GQA ratios 1, 2
and 4, Dk 64 and 128, ragged Dv, conv widths 2..4, padding rows, f32 and bf16,
and a CUDA graph captured once and replayed with new metadata."""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B

pytestmark = pytest.mark.gpu


def make(Bn, Hk, Hv, Dk, Dv, K, dtype, seed, slots=None):
    g0 = torch.Generator().manual_seed(seed)
    C = 2 * Hk * Dk + Hv * Dv
    slots = slots or Bn + 3
    return dict(
        qkvz=torch.randn(Bn, C + Hv * Dv, generator=g0).to(dtype),   # q, k, v then z
        w=torch.randn(C, K, generator=g0) * 0.4,
        ba=torch.randn(Bn, 2 * Hv, generator=g0).to(dtype),          # b then a
        A_log=torch.randn(Hv, generator=g0) * 0.3,
        dt_bias=torch.randn(Hv, generator=g0) * 0.3,
        conv=torch.randn(slots, C, K - 1, generator=g0).to(dtype).float(),
        state=torch.randn(slots, Hv, Dv, Dk, generator=g0) * 0.1,
        idx=torch.randperm(slots, generator=g0)[:Bn].to(torch.int32),
        dims=(Hk, Hv, Dk, Dv, K), C=C)


def gpu(d, dev, conv_d, state_d, idx=None, stream=None):
    Hk, Hv, Dk, Dv, K = d["dims"]
    Bn = d["qkvz"].shape[0]
    ba = d["ba"].to(dev)
    a_raw, b_raw = B.packed_ba_views(ba, Hv)
    out = torch.empty(Bn, Hv, Dv, dtype=d["qkvz"].dtype, device=dev)
    B.gdn_packed_decode(d["qkvz"].to(dev), d["w"].to(dev), a_raw, b_raw, d["A_log"].to(dev),
                        d["dt_bias"].to(dev), (d["idx"] if idx is None else idx).to(dev),
                        conv_d, state_d, out, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K,
                        state_indices_host=d["idx"] if idx is None else None, stream=stream)
    return out


def reference(d, conv, state):
    """O1 (one-token sequences) then O3, f64; beta rounded through b's dtype
    in between ([cpu_ops.cpp] GdnPackedDecodeKernel), nothing else."""
    Hk, Hv, Dk, Dv, K = d["dims"]
    Bn, C = d["qkvz"].shape[0], d["C"]
    x = H.f32(d["qkvz"])[:, :C].astype(np.float64)
    ba = H.f32(d["ba"]).astype(np.float64)
    prep = oracle.prepare_varlen(x, d["w"].numpy(), conv, ba[:, Hv:], ba[:, :Hv],
                                 d["A_log"].numpy(), d["dt_bias"].numpy(),
                                 np.arange(Bn + 1, dtype=np.int32), Hk, Hv, Dk, Dv, K,
                                 state_indices=d["idx"].numpy(), dtype=np.float64)
    if d["ba"].dtype == torch.bfloat16:
        prep["beta"] = H.bf16_round(prep["beta"])
    out = oracle.gdn_decode(prep["q"], prep["k"], prep["v"], prep["g"], prep["beta"], state,
                            1.0 / np.sqrt(Dk), state_indices=d["idx"].numpy(), dtype=np.float64)
    return out


def run(Bn, Hk, Hv, Dk, Dv, K, dtype, dev, seed, edit=None):
    d = make(Bn, Hk, Hv, Dk, Dv, K, dtype, seed)
    if edit is not None:
        edit(d)
    conv_ref = d["conv"].numpy().astype(np.float64).copy()
    state_ref = d["state"].numpy().astype(np.float64).copy()
    conv_d, state_d = d["conv"].to(dev), d["state"].to(dev)
    out = gpu(d, dev, conv_d, state_d)
    B.gdn_read_device_status()
    ref_out = reference(d, conv_ref, state_ref)
    tol = H.TOL_F32 if dtype == torch.float32 else H.TOL_BF16
    H.check(out, ref_out, tol, "packed decode out")
    H.assert_close(H.f32(state_d), state_ref, tol, "packed decode state")
    np.testing.assert_array_equal(H.f32(conv_d), conv_ref.astype(np.float32))
    return d


def test_packed_decode_b256_shape(cuda_device):
    run(256, 16, 32, 128, 128, 4, torch.bfloat16, cuda_device, seed=1)


@pytest.mark.parametrize("Hk,Hv,Dk,Dv,K", [(4, 4, 128, 128, 4), (2, 8, 128, 64, 3),
                                           (4, 8, 64, 96, 2), (1, 2, 64, 40, 4)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_packed_decode_shapes(Hk, Hv, Dk, Dv, K, dtype, cuda_device):
    run(33, Hk, Hv, Dk, Dv, K, dtype, cuda_device, seed=Hk * 100 + Hv + Dv + K)


def test_packed_decode_padding_rows(cuda_device):
    def edit(d):
        d["idx"][[0, 5, 6]] = -1
    run(12, 2, 4, 128, 128, 4, torch.bfloat16, cuda_device, seed=3, edit=edit)


def test_packed_decode_cuda_graph_replay(cuda_device):
    """A fixed 64-row batch is captured once; each replay runs different rows
    (the rest padded with -1) on the same slots' evolving states."""
    dev = cuda_device
    d = make(64, 4, 8, 128, 128, 4, torch.bfloat16, 4, slots=80)
    conv_d, state_d = d["conv"].to(dev), d["state"].to(dev)
    conv_ref = d["conv"].numpy().astype(np.float64).copy()
    state_ref = d["state"].numpy().astype(np.float64).copy()
    idx_d = torch.full((64,), -1, dtype=torch.int32, device=dev)
    B.gdn_packed_decode(d["qkvz"].to(dev)[:1], d["w"].to(dev), *B.packed_ba_views(
        d["ba"].to(dev)[:1], 8), d["A_log"].to(dev), d["dt_bias"].to(dev), idx_d[:1], conv_d,
        state_d, torch.empty(1, 8, 128, dtype=torch.bfloat16, device=dev), Hk=4, Hv=8, Dk=128,
        Dv=128, K=4)                                   # first call outside the capture
    torch.cuda.synchronize()
    # every tensor the graph reads is allocated before the capture
    x_d, ba_d = d["qkvz"].to(dev), d["ba"].to(dev)
    w_d, alog_d, dtb_d = d["w"].to(dev), d["A_log"].to(dev), d["dt_bias"].to(dev)
    a_v, b_v = B.packed_ba_views(ba_d, 8)
    out_d = torch.empty(64, 8, 128, dtype=torch.bfloat16, device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.gdn_packed_decode(x_d, w_d, a_v, b_v, alog_d, dtb_d, idx_d, conv_d, state_d, out_d,
                            Hk=4, Hv=8, Dk=128, Dv=128, K=4, stream=torch.cuda.current_stream())
    g1 = torch.Generator().manual_seed(5)
    for live in (40, 64, 7):
        idx = torch.full((64,), -1, dtype=torch.int32)
        idx[:live] = torch.randperm(80, generator=g1)[:live].to(torch.int32)
        idx_d.copy_(idx)
        graph.replay()
        torch.cuda.synchronize()
        B.gdn_read_device_status()
        step = dict(d, idx=idx)
        ref = reference(step, conv_ref, state_ref)
        H.check(out_d, ref, H.TOL_BF16, f"graph replay {live}")
    H.assert_close(H.f32(state_d), state_ref, H.TOL_BF16, "graph replay states")
    np.testing.assert_array_equal(H.f32(conv_d), conv_ref.astype(np.float32))
