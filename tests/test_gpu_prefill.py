"""GPU parity of gdn_prefill_varlen against the oracle's sequential recurrence (O2).

Every algorithm (the chunked tensor-core form in one fused launch and in two
launches with a workspace, where supported, and the token-sequential recurrent
form everywhere) is checked on: ragged varlen batches whose lengths
straddle the chunk size (1, 63, 64, 65, 127, 128, 129, ...), batches the
two-launch form takes in pieces of chunk indices, padding slots,
has_initial_state mixes, GQA ratios, f32 and bf16, in-kernel q/k norm, the
weak-decay twins (slow decay, so a wrong carried state is not hidden), and the
prefill workloads at full size (outputs of every head for the single 4096-token
sequence, and every sequence and head of the 8-sequence varlen batch).
Inputs are the oracle's prepare outputs rounded to the activation dtype by
torch; the oracle gets the same rounded values.
"""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B
from gated_delta_rule_44_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ALGOS = (B.GDN_PREFILL_RECURRENT, B.GDN_PREFILL_CHUNKED, B.GDN_PREFILL_FUSED)


def algo_ok(algo, w):
    """The tensor-core algorithms are built for bf16 with Dk = Dv = 128."""
    if algo == B.GDN_PREFILL_RECURRENT:
        return True
    dt = B.GDN_DTYPE_BF16 if w.act_dtype == torch.bfloat16 else B.GDN_DTYPE_F32
    return B.gdn_prefill_resolve_algo(w.N, w.Hv, w.Dk, w.Dv, dt) != B.GDN_PREFILL_RECURRENT


def run_prefill(w, dev, algo, seqs=None, heads=None, norm=False, scale=-1.0, host=True):
    ref_prep, _ = H.oracle_prepare(w, norm=not norm)
    acts = {k: torch.from_numpy(ref_prep[k]).to(w.act_dtype) for k in ("q", "k", "v")}
    g = torch.from_numpy(ref_prep["g"])
    beta = torch.from_numpy(ref_prep["beta"])
    out = torch.full((w.T, w.Hv, w.Dv), float("nan"), dtype=w.act_dtype, device=dev)
    pool = w.state_pool.to(dev)
    dt = B.GDN_DTYPE_BF16 if w.act_dtype == torch.bfloat16 else B.GDN_DTYPE_F32
    ws_bytes = B.gdn_prefill_workspace_bytes(w.T, w.N, w.Hv, w.Dk, w.Dv, dt, algo)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    B.gdn_prefill_varlen(acts["q"].to(dev), acts["k"].to(dev), acts["v"].to(dev), g.to(dev),
                         beta.to(dev), pool, w.cu_seqlens.to(dev), out, scale=scale,
                         state_indices=w.state_indices.to(dev),
                         has_initial_state=w.has_initial_state.to(dev),
                         cu_seqlens_host=w.cu_seqlens if host else None,
                         state_indices_host=w.state_indices if host else None,
                         use_qk_l2norm=norm, algo=algo, workspace=ws)
    B.gdn_read_device_status()
    seqs = list(range(w.N)) if seqs is None else seqs
    heads = list(range(w.Hv)) if heads is None else heads
    cpool, remap = H.compact_pool(w, seqs)
    items = H.seq_head_items(w, seqs, heads)
    sc = scale if scale >= 0 else 1.0 / np.sqrt(w.Dk)
    ref_out = oracle.gdn_varlen(H.f32(acts["q"]), H.f32(acts["k"]), H.f32(acts["v"]), g.numpy(),
                                beta.numpy(), cpool, w.cu_seqlens.numpy(), sc,
                                state_indices=remap, has_initial_state=w.has_initial_state.numpy(),
                                use_qk_l2norm=norm, items=items, dtype=np.float32)
    tol = H.tol_for(w)
    cu = w.cu_seqlens.tolist()
    got = H.f32(out)
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])
    e_out = H.assert_close(got[rows][:, heads], ref_out[rows][:, heads], tol, "out",
                           stored_bf16=w.act_dtype == torch.bfloat16)
    got_pool = H.f32(pool)
    live = [s for s in seqs if remap[s] >= 0]
    e_state = 0.0
    if live:
        gp = np.stack([got_pool[int(w.state_indices[s])][heads] for s in live])
        rp = np.stack([cpool[remap[s]][heads] for s in live])
        e_state = H.assert_close(gp, rp, tol, "state")
    if len(seqs) == w.N and len(heads) == w.Hv:
        used = {int(s) for s in w.state_indices.tolist() if s >= 0}
        for slot in range(w.slots):
            if slot not in used:
                np.testing.assert_array_equal(got_pool[slot], w.state_pool[slot].numpy())
    return e_out, e_state


SMALL = [
    # seqlens, Hk, Hv, Dk, Dv, dtype, padded, prefill_new, weak
    ([64], 2, 4, 32, 32, torch.float32, None, True, False),
    ([1, 63, 64, 65, 2, 127], 2, 4, 32, 32, torch.float32, [3], False, True),
    ([1, 63, 64, 65, 2, 127], 2, 4, 128, 128, torch.bfloat16, [3], False, True),
    ([129, 128, 3, 200], 1, 4, 128, 128, torch.bfloat16, None, True, True),
    ([129, 128, 3, 200], 2, 2, 128, 128, torch.bfloat16, None, False, False),
    ([300, 5], 2, 4, 64, 64, torch.bfloat16, None, False, True),
    ([40, 9, 17], 2, 6, 16, 24, torch.float32, [1], False, True),
    # eight value heads per key head: chunk_prep's loop over a key head's heads
    ([100, 37, 64, 1], 1, 8, 128, 128, torch.bfloat16, [1], False, True),
    # few chains and more than 16 chunks: the two-launch form runs in pieces of
    # chunk indices (each piece's scan resumes from the state the previous one
    # stored, fresh sequences included), with a padded sequence
    ([1030, 64, 1, 700], 2, 4, 128, 128, torch.bfloat16, [2], False, True),
    ([1030, 64, 1, 700], 2, 4, 128, 128, torch.bfloat16, [1], True, False),
]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_prefill_small(case, algo, cuda_device):
    seqlens, Hk, Hv, Dk, Dv, dt, padded, new, weak = SMALL[case]
    w = W.make_workload("p", 300 + case, seqlens, Hk, Hv, Dk, Dv, act_dtype=dt,
                        slots=len(seqlens) + 2, padded=padded, prefill_new=new, n_decode=0,
                        weak_decay=weak, state_std=0.3)
    if not algo_ok(algo, w):
        pytest.skip("algorithm not built for these dims")
    run_prefill(w, cuda_device, algo)


@pytest.mark.parametrize("algo", ALGOS)
def test_prefill_norm_scale_no_mirrors(algo, cuda_device):
    w = W.make_workload("p", 320, [70, 1, 64], 2, 4, 128, 128, act_dtype=torch.bfloat16,
                        weak_decay=True, state_std=0.3)
    if not algo_ok(algo, w):
        pytest.skip("algorithm not built for these dims")
    run_prefill(w, cuda_device, algo, norm=True, scale=0.2, host=False)


@pytest.mark.parametrize("weak", [False, True])
@pytest.mark.parametrize("algo", ALGOS)
def test_prefill_4k_full_size(algo, weak, cuda_device):
    w = W.named("prefill_4k", weak_decay=weak)
    if not algo_ok(algo, w):
        pytest.skip("algorithm not built for these dims")
    e = run_prefill(w, cuda_device, algo)
    print(f"prefill_4k algo={algo} weak={weak}: out err {e[0]:.2e}, state err {e[1]:.2e}")


@pytest.mark.parametrize("weak", [False, True])
@pytest.mark.parametrize("algo", ALGOS)
def test_varlen_8_full_size(algo, weak, cuda_device):
    """Every sequence and every value head of the 8-sequence varlen workload
    (the oracle runs on all host cores)."""
    w = W.named("varlen_8", weak_decay=weak)
    if not algo_ok(algo, w):
        pytest.skip("algorithm not built for these dims")
    e = run_prefill(w, cuda_device, algo)
    print(f"varlen_8 algo={algo} weak={weak}: out err {e[0]:.2e}, state err {e[1]:.2e}")


SPREAD = [
    # more chains than SMs, so the fused form spreads the chains' chunks over
    # gangs of Hv / Hk CTAs, one CTA per SM (chains cut between two gangs
    # resume from the state the other stored): decodes, ragged new prefills,
    # padding
    ([1] * 10 + [int(x) for x in np.random.default_rng(5).integers(2, 400, 35)], [3, 20], 2, 4),
    # one sequence longer than the even share: every gang's range is its length
    ([3000] + [int(x) for x in np.random.default_rng(6).integers(1, 200, 47)], [9], 2, 4),
    # gangs of 3 (152 SMs leave 2 CTAs without a range) and of 8
    ([1] * 10 + [int(x) for x in np.random.default_rng(7).integers(2, 700, 20)], [12], 2, 6),
    ([1] * 10 + [int(x) for x in np.random.default_rng(8).integers(2, 900, 10)], [], 1, 8),
]


@pytest.mark.parametrize("case", range(len(SPREAD)))
def test_fused_spread_over_sms(case, cuda_device):
    """The fused form with its workspace (chunks spread over the SMs) against
    the oracle, and bit for bit against the same call without the workspace
    (one CTA per chain): a chain's state crosses CTAs through the pool in f32,
    so the arithmetic does not change."""
    seqlens, padded, Hk, Hv = SPREAD[case]
    w = W.make_workload("p", 340 + case, seqlens, Hk, Hv, 128, 128, act_dtype=torch.bfloat16,
                        slots=len(seqlens) + 2, padded=padded, prefill_new=True, n_decode=10,
                        weak_decay=True, state_std=0.3)
    assert w.N * w.Hv > torch.cuda.get_device_properties(cuda_device).multi_processor_count
    run_prefill(w, cuda_device, B.GDN_PREFILL_FUSED)
    ref_prep, _ = H.oracle_prepare(w, norm=True)
    dev = cuda_device
    args = [torch.from_numpy(ref_prep[k]).to(w.act_dtype).to(dev) for k in ("q", "k", "v")]
    args += [torch.from_numpy(ref_prep[k]).to(dev) for k in ("g", "beta")]
    ws_bytes = B.gdn_prefill_workspace_bytes(w.T, w.N, w.Hv, w.Dk, w.Dv, B.GDN_DTYPE_BF16,
                                             B.GDN_PREFILL_FUSED)
    assert ws_bytes > 0
    results = []
    for ws, launches in ((torch.empty(ws_bytes, dtype=torch.uint8, device=dev), 2), (None, 1)):
        pool = w.state_pool.to(dev)
        out = torch.full((w.T, w.Hv, w.Dv), float("nan"), dtype=w.act_dtype, device=dev)
        n0 = B.gdn_launch_count()
        B.gdn_prefill_varlen(*args, pool, w.cu_seqlens.to(dev), out,
                             state_indices=w.state_indices.to(dev),
                             has_initial_state=w.has_initial_state.to(dev),
                             algo=B.GDN_PREFILL_FUSED, workspace=ws)
        # the ranges run as the schedule kernel and the fused kernel; without
        # the workspace the fused kernel alone runs one CTA per chain
        assert B.gdn_launch_count() - n0 == launches
        B.gdn_read_device_status()
        results.append((out, pool))
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1])


def test_fused_spread_cuda_graph_replay(cuda_device):
    """The spread fused form (its schedule kernel, then a cooperative launch)
    captured in a CUDA graph: replays match eager calls bit for bit."""
    dev = cuda_device
    w = W.make_workload("p", 350, [int(x) for x in np.random.default_rng(9).integers(1, 300, 45)],
                        2, 4, 128, 128, act_dtype=torch.bfloat16, weak_decay=True, state_std=0.3)
    assert w.N * w.Hv > torch.cuda.get_device_properties(dev).multi_processor_count
    ref_prep, _ = H.oracle_prepare(w, norm=True)
    args = [torch.from_numpy(ref_prep[k]).to(w.act_dtype).to(dev) for k in ("q", "k", "v")]
    args += [torch.from_numpy(ref_prep[k]).to(dev) for k in ("g", "beta")]
    ws = torch.empty(B.gdn_prefill_workspace_bytes(w.T, w.N, w.Hv, w.Dk, w.Dv, B.GDN_DTYPE_BF16,
                                                   B.GDN_PREFILL_FUSED),
                     dtype=torch.uint8, device=dev)
    cu, sidx, hi = (x.to(dev) for x in (w.cu_seqlens, w.state_indices, w.has_initial_state))
    pool0 = w.state_pool.to(dev)
    pe, pg = pool0.clone(), pool0.clone()
    oe = torch.empty((w.T, w.Hv, w.Dv), dtype=w.act_dtype, device=dev)
    og = torch.empty_like(oe)

    def call(pool, out, stream=None):
        B.gdn_prefill_varlen(*args, pool, cu, out, state_indices=sidx, has_initial_state=hi,
                             algo=B.GDN_PREFILL_FUSED, workspace=ws, stream=stream)

    call(pool0.clone(), torch.empty_like(oe))  # settles the host-side resources
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(pg, og, stream=torch.cuda.current_stream())
    for _ in range(3):
        call(pe, oe)
        graph.replay()
        torch.cuda.synchronize()
        B.gdn_read_device_status()
        assert torch.equal(oe, og)
        assert torch.equal(pe, pg)
