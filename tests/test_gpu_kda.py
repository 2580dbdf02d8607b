"""GPU parity of gdn_kda_varlen (the gated delta rule with one log decay per
key channel, [cpu_ops.cpp] KdaHeadTokenStep / KdaGatedDeltaRuleKernel) against
the oracle's KDA chain, through the C ABI: varlen prefill, decode (one-token
sequences), padding slots, fresh states, bf16 and f32, every supported Dk; the
chunked tensor-core form at chunk-boundary lengths, strong and weak decays,
GQA, padding and fresh states, and the single-sequence prefill shape at full
size (4096 tokens, 16 / 32 heads of 128)."""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B

pytestmark = pytest.mark.gpu


def run(seqs, Hk, Hv, Dk, Dv, dtype, dev, seed, sidx=None, has_init=None, slots=None,
        algo=B.GDN_PREFILL_AUTO, g_scale=0.3):
    g0 = torch.Generator().manual_seed(seed)
    T, N = sum(seqs), len(seqs)
    slots = slots or N + 2
    cu = torch.tensor(np.concatenate([[0], np.cumsum(seqs)]), dtype=torch.int32)
    q = (torch.randn(T, Hk, Dk, generator=g0) / np.sqrt(Dk)).to(dtype)
    k = (torch.randn(T, Hk, Dk, generator=g0) / np.sqrt(Dk)).to(dtype)
    v = torch.randn(T, Hv, Dv, generator=g0).to(dtype)
    g = -torch.rand(T, Hv, Dk, generator=g0) * g_scale      # log decay per key channel
    beta = torch.rand(T, Hv, generator=g0) * 0.8 + 0.1
    pool = torch.randn(slots, Hv, Dv, Dk, generator=g0) * 0.1
    if sidx is None:
        sidx = torch.randperm(slots, generator=g0)[:N].to(torch.int32)
    hi = None if has_init is None else torch.tensor(has_init, dtype=torch.uint8)
    out = torch.empty(T, Hv, Dv, dtype=dtype, device=dev)
    pool_d = pool.to(dev)
    B.gdn_kda_varlen(q.to(dev), k.to(dev), v.to(dev), g.to(dev), beta.to(dev), pool_d,
                     cu.to(dev), out, scale=-1.0, state_indices=sidx.to(dev),
                     has_initial_state=None if hi is None else hi.to(dev),
                     cu_seqlens_host=cu, state_indices_host=sidx, algo=algo)
    B.gdn_read_device_status()
    torch.cuda.synchronize()
    ref_pool = pool.numpy().astype(np.float32).copy()
    ref = oracle.kda_varlen(H.f32(q), H.f32(k), H.f32(v), g.numpy(), beta.numpy(), ref_pool,
                            cu.numpy(), 1.0 / np.sqrt(Dk), state_indices=sidx.numpy(),
                            has_initial_state=None if hi is None else hi.numpy(),
                            dtype=np.float32)
    tol = H.TOL_F32 if dtype == torch.float32 else H.TOL_BF16
    H.check(out, ref, tol, "kda out")
    H.assert_close(H.f32(pool_d), ref_pool, tol, "kda state")
    return out, pool_d


@pytest.mark.parametrize("Dk", [16, 32, 64, 128, 256])
def test_kda_varlen_all_dk(Dk, cuda_device):
    run([7, 1, 70], 2, 4, Dk, 64, torch.bfloat16, cuda_device, seed=Dk)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_kda_decode_rows(dtype, cuda_device):
    run([1] * 33, 2, 4, 128, 128, dtype, cuda_device, seed=3)


def test_kda_padding_and_fresh_states(cuda_device):
    run([5, 3, 9, 2], 1, 2, 128, 32, torch.float32, cuda_device, seed=4,
        sidx=torch.tensor([2, -1, 0, 5], dtype=torch.int32), has_init=[1, 1, 0, 1], slots=6)


def test_kda_long_sequence(cuda_device):
    run([1000], 4, 8, 128, 128, torch.bfloat16, cuda_device, seed=5, algo=B.GDN_PREFILL_RECURRENT)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_kda_decode_form_padding_and_fresh_states(dtype, cuda_device):
    # T == N runs the decode form: padding rows and has_initial_state = 0 there
    run([1] * 9, 2, 4, 128, 96, dtype, cuda_device, seed=6,
        sidx=torch.tensor([3, -1, 0, 8, 5, -1, 1, 2, 7], dtype=torch.int32),
        has_init=[1, 1, 0, 1, 0, 1, 1, 1, 0], slots=10)


CHUNKED = B.GDN_PREFILL_CHUNKED


def test_kda_chunked_chunk_boundaries(cuda_device):
    run([1, 63, 64, 65, 127, 128, 129], 2, 4, 128, 128, torch.bfloat16, cuda_device, seed=11,
        algo=CHUNKED)


@pytest.mark.parametrize("g_scale", [6.0, 0.02])
def test_kda_chunked_strong_and_weak_decay(g_scale, cuda_device):
    """Per-token decays down to e^-6 per channel (products underflow within a
    sub-chunk) and nearly none (the state keeps its whole history)."""
    run([200, 77, 130], 2, 8, 128, 128, torch.bfloat16, cuda_device, seed=12, algo=CHUNKED,
        g_scale=g_scale)


def test_kda_chunked_padding_and_fresh_states(cuda_device):
    run([70, 3, 129, 64], 1, 4, 128, 128, torch.bfloat16, cuda_device, seed=13, algo=CHUNKED,
        sidx=torch.tensor([2, -1, 0, 5], dtype=torch.int32), has_init=[1, 1, 0, 1], slots=6)


def test_kda_chunked_single_token_sequences(cuda_device):
    """T == N on the chunked form: every chunk is one token long."""
    run([1] * 9, 2, 4, 128, 128, torch.bfloat16, cuda_device, seed=14, algo=CHUNKED)


def test_kda_chunked_matches_recurrent(cuda_device):
    """Both GPU forms against the oracle, and against each other."""
    o1, s1 = run([1000, 37], 4, 8, 128, 128, torch.bfloat16, cuda_device, seed=15, algo=CHUNKED)
    o2, s2 = run([1000, 37], 4, 8, 128, 128, torch.bfloat16, cuda_device, seed=15,
                 algo=B.GDN_PREFILL_RECURRENT)
    e = H.rel_err_stored_bf16(H.f32(o1), H.f32(o2))
    assert e <= H.TOL_BF16, f"chunked vs recurrent out {e:.3e}"


def test_kda_chunked_full_size(cuda_device):
    """The single-sequence prefill shape: 4096 tokens, Hk = 16, Hv = 32, D = 128."""
    run([4096], 16, 32, 128, 128, torch.bfloat16, cuda_device, seed=16, algo=CHUNKED)


def test_kda_chunked_pieces_padding_and_fresh_states(cuda_device):
    """Few chains and more than 16 chunks: the chunked form runs in pieces of
    chunk indices (here 64 chains leave 88 SMs, so 8 chunk indices a piece and
    3 pieces); later pieces resume from the state the previous piece stored (a
    fresh sequence included), a padded sequence stays untouched."""
    run([1100, 5, 300, 77], 4, 16, 128, 128, torch.bfloat16, cuda_device, seed=17, algo=CHUNKED,
        sidx=torch.tensor([4, -1, 0, 2], dtype=torch.int32), has_init=[0, 1, 1, 0], slots=6)


def test_kda_chunked_pieces_cuda_graph_replay(cuda_device):
    """The chunked KDA form in pieces (programmatic dependent launches; 64
    chains, 3 pieces of 8 chunk indices) captured in a CUDA graph: replays
    match eager calls bit for bit."""
    dev = cuda_device
    g0 = torch.Generator().manual_seed(18)
    lens = [1100, 300]
    T, N, Hk, Hv, D = sum(lens), len(lens), 8, 32, 128
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    q = (torch.randn(T, Hk, D, generator=g0) / np.sqrt(D)).to(torch.bfloat16).to(dev)
    k = (torch.randn(T, Hk, D, generator=g0) / np.sqrt(D)).to(torch.bfloat16).to(dev)
    v = torch.randn(T, Hv, D, generator=g0).to(torch.bfloat16).to(dev)
    g = (-torch.rand(T, Hv, D, generator=g0) * 0.3).to(dev)
    beta = (torch.rand(T, Hv, generator=g0) * 0.8 + 0.1).to(dev)
    pool0 = torch.randn(N, Hv, D, D, generator=g0).to(dev) * 0.1
    ws = torch.empty(B.gdn_kda_workspace_bytes(T, N, Hv, D, D, 1, CHUNKED), dtype=torch.uint8,
                     device=dev)
    pe, pg = pool0.clone(), pool0.clone()
    oe = torch.empty(T, Hv, D, dtype=torch.bfloat16, device=dev)
    og = torch.empty_like(oe)

    def call(pool, out, stream=None):
        B.gdn_kda_varlen(q, k, v, g, beta, pool, cu, out, algo=CHUNKED, workspace=ws,
                         stream=stream)

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
