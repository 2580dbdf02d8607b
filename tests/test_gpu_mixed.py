"""End-to-end GPU parity of one mixed serving step (prepare, then decode on the
leading single-token rows and the prefill on the rest) against the oracle's
prepare + sequential recurrence from the same raw inputs.

The GPU stores q, k, v and out in bf16; the oracle's q, k, v are rounded to
bf16 between its two steps in the same way (the pages' store convention) and
`out` is compared with the bf16-storage metric of tests/helpers.py, plus the
oracle's bound on what a one-step rounding flip of a near-boundary q, k or v
value can carry into the outputs.  The full-size mixed workload
(512 decodes + 4 x 2048-token prefills, Hv = 64, 1024-slot pool) is compared on
every row and head, plus the whole conv pool.
"""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B
from gated_delta_rule_44_gb300 import layer
from gated_delta_rule_44_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_mixed(w, dev, seqs, heads):
    d = H.to_dev(w, dev)
    out = layer.mixed_step(d["mixed_qkv"], d["a_raw"], d["b_raw"], d["conv_weight"], d["A_log"],
                           d["dt_bias"], d["cu_seqlens"], d["state_indices"],
                           d["has_initial_state"], d["state_pool"], d["conv_pool"],
                           n_decode=w.n_decode, Hk=w.Hk, Hv=w.Hv, Dk=w.Dk, Dv=w.Dv, K=w.K,
                           cu_seqlens_prefill=d["cu_seqlens_prefill"])
    torch.cuda.synchronize()
    ref_prep, ref_conv = H.oracle_prepare(w)
    cpool, remap = H.compact_pool(w, seqs)
    # Where the path's and the oracle's f32 q, k, v may round to neighbouring
    # bf16 values, the outputs may differ by that step carried through the
    # recurrence: the oracle bounds it (tests/helpers.py, stored_flip_bound).
    extra, extra_state = H.stored_flip_bound(ref_prep, w.cu_seqlens.numpy(), 1.0 / np.sqrt(w.Dk),
                                             cpool, state_indices=remap,
                                             has_initial_state=w.has_initial_state.numpy())
    # the path stores q, k, v in bf16 between the two steps, as the pages do
    for key in ("q", "k", "v"):
        ref_prep[key] = H.bf16_round(ref_prep[key]).astype(np.float32)
    items = H.seq_head_items(w, seqs, heads)
    ref_out = oracle.gdn_varlen(ref_prep["q"], ref_prep["k"], ref_prep["v"], ref_prep["g"],
                                ref_prep["beta"], cpool, w.cu_seqlens.numpy(),
                                1.0 / np.sqrt(w.Dk), state_indices=remap,
                                has_initial_state=w.has_initial_state.numpy(), items=items,
                                dtype=np.float32)
    cu = w.cu_seqlens.tolist()
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])
    tol = H.tol_for(w)
    e_out = H.assert_close(H.f32(out)[rows][:, heads], ref_out[rows][:, heads], tol, "out",
                           stored_bf16=True, extra=extra[rows][:, heads])
    gp = d["state_pool"]
    live = [s for s in seqs if remap[s] >= 0]
    e_state = H.assert_close_blocks(
        ((H.f32(gp[int(w.state_indices[s])][heads]), cpool[remap[s]][heads],
          extra_state[remap[s]][heads][..., None]) for s in live),
        tol, "state")
    np.testing.assert_array_equal(H.f32(d["conv_pool"]), ref_conv)
    return e_out, e_state


@pytest.mark.parametrize("weak", [False, True])
def test_mixed_small(weak, cuda_device):
    w = W.make_workload("m", 400, [1] * 9 + [70, 129, 3], 2, 4, 128, 128, slots=20, n_decode=9,
                        prefill_new=True, padded=[4], weak_decay=weak, state_std=0.3)
    run_mixed(w, cuda_device, list(range(w.N)), list(range(w.Hv)))


def test_mixed_hv64_full_size(cuda_device):
    """All 512 decode rows and all 4 prefills, every one of the 64 value heads."""
    w = W.named("mixed_hv64")
    e = run_mixed(w, cuda_device, list(range(w.N)), list(range(w.Hv)))
    print(f"mixed_hv64: out err {e[0]:.2e}, state err {e[1]:.2e}")


def test_host_pipeline_matches_sequential_steps(cuda_device):
    """GdnHostPipeline (inputs copied in and outputs copied out on their own
    streams, overlapping the neighbouring steps' compute) gives bit-identical
    outputs, state and conv pools to the same steps run one after another."""
    w = W.make_workload("pipe", 402, [1] * 5 + [70, 129], 2, 4, 128, 128, slots=12, n_decode=5,
                        prefill_new=True, state_std=0.3)
    steps = 3
    # per-step inputs differ: a fresh mixed_qkv per step
    gen = torch.Generator().manual_seed(11)
    xs = [torch.randn(w.mixed_qkv.shape, generator=gen).to(w.mixed_qkv.dtype) for _ in range(steps)]

    def make_step(d):
        return layer.GdnStep(w.T, w.N, w.n_decode, w.Hk, w.Hv, w.Dk, w.Dv, w.K, w.act_dtype,
                             cuda_device)

    # sequential reference on the device
    d1 = H.to_dev(w, cuda_device)
    st1 = make_step(d1)
    ref_out = []
    for x in xs:
        o = st1.run(x.to(cuda_device), d1["a_raw"], d1["b_raw"], d1["conv_weight"], d1["A_log"],
                    d1["dt_bias"], d1["cu_seqlens"], d1["state_indices"], d1["has_initial_state"],
                    d1["state_pool"], d1["conv_pool"], d1["cu_seqlens_prefill"])
        ref_out.append(o.clone())
    torch.cuda.synchronize()

    # pipelined from pinned host memory
    d2 = H.to_dev(w, cuda_device)
    pipe = layer.GdnHostPipeline(make_step(d2), cuda_device)
    host_outs = [torch.empty(w.T, w.Hv, w.Dv, dtype=w.act_dtype).pin_memory() for _ in range(steps)]
    for x, ho in zip(xs, host_outs):
        host_in = {"mixed_qkv": x.pin_memory(), "a_raw": w.a_raw.pin_memory(),
                   "b_raw": w.b_raw.pin_memory(), "cu_seqlens": w.cu_seqlens.pin_memory(),
                   "state_indices": w.state_indices.pin_memory(),
                   "has_initial_state": w.has_initial_state.pin_memory(),
                   "cu_seqlens_prefill": w.cu_seqlens_prefill.pin_memory()}
        pipe.submit(host_in, ho, d2["conv_weight"], d2["A_log"], d2["dt_bias"], d2["state_pool"],
                    d2["conv_pool"])
    pipe.synchronize()
    for r, ho in zip(ref_out, host_outs):
        assert torch.equal(r.cpu(), ho)
    assert torch.equal(d1["state_pool"], d2["state_pool"])
    assert torch.equal(d1["conv_pool"], d2["conv_pool"])


def test_mixed_step_cuda_graph_replay(cuda_device):
    """A whole mixed step (prepare, decode, chunked prefill) captured once in
    a CUDA graph and replayed gives bit-identical outputs, state and conv pools
    to the same steps run eagerly: the host validation, the status-word lookup
    and the prefill's tensor maps are all settled before the capture."""
    dev = cuda_device
    w = W.make_workload("graph", 403, [1] * 6 + [100, 64, 3], 2, 4, 128, 128, slots=14,
                        n_decode=6, prefill_new=False, state_std=0.3)
    eager, graphed = H.to_dev(w, dev), H.to_dev(w, dev)
    step_e = layer.GdnStep(w.T, w.N, w.n_decode, w.Hk, w.Hv, w.Dk, w.Dv, w.K, w.act_dtype, dev)
    step_g = layer.GdnStep(w.T, w.N, w.n_decode, w.Hk, w.Hv, w.Dk, w.Dv, w.K, w.act_dtype, dev)

    def run(step, d, stream=None):
        return step.run(d["mixed_qkv"], d["a_raw"], d["b_raw"], d["conv_weight"], d["A_log"],
                        d["dt_bias"], d["cu_seqlens"], d["state_indices"],
                        d["has_initial_state"], d["state_pool"], d["conv_pool"],
                        d["cu_seqlens_prefill"], stream=stream)

    # a throw-away eager step on copies settles every lazy host-side resource
    warm = H.to_dev(w, dev)
    run(step_g, warm)
    torch.cuda.synchronize()
    del warm
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(step_g, graphed, stream=torch.cuda.current_stream())
    for _ in range(2):
        run(step_e, eager)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(step_e.out, step_g.out)
        assert torch.equal(eager["state_pool"], graphed["state_pool"])
        assert torch.equal(eager["conv_pool"], graphed["conv_pool"])


def test_pieces_cuda_graph_replay(cuda_device):
    """A mixed step whose prefill takes the two-launch form in pieces chained
    by programmatic dependent launch (2 prefill sequences x 4 heads, 21
    chunks), captured in a CUDA graph: replays match eager steps bit for bit."""
    dev = cuda_device
    w = W.make_workload("graph", 404, [1, 1, 1100, 200], 2, 4, 128, 128, slots=7,
                        n_decode=2, prefill_new=False, state_std=0.3)
    assert B.gdn_prefill_resolve_algo(2, 4, 128, 128) == B.GDN_PREFILL_CHUNKED
    eager, graphed = H.to_dev(w, dev), H.to_dev(w, dev)
    step_e = layer.GdnStep(w.T, w.N, w.n_decode, w.Hk, w.Hv, w.Dk, w.Dv, w.K, w.act_dtype, dev)
    step_g = layer.GdnStep(w.T, w.N, w.n_decode, w.Hk, w.Hv, w.Dk, w.Dv, w.K, w.act_dtype, dev)

    def run(step, d, stream=None):
        return step.run(d["mixed_qkv"], d["a_raw"], d["b_raw"], d["conv_weight"], d["A_log"],
                        d["dt_bias"], d["cu_seqlens"], d["state_indices"],
                        d["has_initial_state"], d["state_pool"], d["conv_pool"],
                        d["cu_seqlens_prefill"], stream=stream)

    warm = H.to_dev(w, dev)
    run(step_g, warm)
    torch.cuda.synchronize()
    del warm
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(step_g, graphed, stream=torch.cuda.current_stream())
    for _ in range(3):
        run(step_e, eager)
        graph.replay()
        torch.cuda.synchronize()
        B.gdn_read_device_status()
        assert torch.equal(step_e.out, step_g.out)
        assert torch.equal(eager["state_pool"], graphed["state_pool"])
        assert torch.equal(eager["conv_pool"], graphed["conv_pool"])
