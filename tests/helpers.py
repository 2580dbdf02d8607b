"""Shared test helpers: run the CUDA path and the oracle on the same seeded
workload and compare them.

The parity metric is the one the layer is specified with:
    err = max |gpu - ref| / rms(ref)
over the whole compared tensor, with tolerance 1e-4 for f32 activations and
2e-2 for bf16 activations (state always f32).  Oracle inputs come only from the
workload generator (bf16 values widened exactly to f32) or from the oracle's
own earlier steps, never from the CUDA path.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_delta_rule_44_gb300 import binding as B
from gated_delta_rule_44_gb300.workloads import Workload

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def tol_for(w: Workload) -> float:
    return TOL_F32 if w.act_dtype == torch.float32 else TOL_BF16


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt((ref ** 2).mean()))
    diff = float(np.abs(gpu - ref).max())
    if rms == 0.0:
        return diff
    return diff / rms


def assert_close(gpu, ref, tol, what=""):
    e = rel_err(gpu, ref)
    assert np.all(np.isfinite(np.asarray(gpu, dtype=np.float64))), f"{what}: non-finite"
    assert e <= tol, f"{what}: max|err|/rms(ref) = {e:.3e} > {tol:.1e}"
    return e


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


# ---- CUDA path -----------------------------------------------------------------

def to_dev(w: Workload, dev):
    """Device copies of every input of the workload (the pools are copied too)."""
    return dict(
        mixed_qkv=w.mixed_qkv.to(dev), conv_weight=w.conv_weight.to(dev), a_raw=w.a_raw.to(dev),
        b_raw=w.b_raw.to(dev), A_log=w.A_log.to(dev), dt_bias=w.dt_bias.to(dev),
        cu_seqlens=w.cu_seqlens.to(dev), state_indices=w.state_indices.to(dev),
        has_initial_state=w.has_initial_state.to(dev), state_pool=w.state_pool.to(dev),
        conv_pool=w.conv_pool.to(dev), cu_seqlens_prefill=w.cu_seqlens_prefill.to(dev))


def gpu_prepare(w: Workload, d, norm=True, host_mirrors=True):
    dev = d["mixed_qkv"].device
    T = w.T
    q = torch.empty((T, w.Hk, w.Dk), dtype=w.act_dtype, device=dev)
    k = torch.empty_like(q)
    v = torch.empty((T, w.Hv, w.Dv), dtype=w.act_dtype, device=dev)
    g = torch.empty((T, w.Hv), dtype=torch.float32, device=dev)
    beta = torch.empty_like(g)
    B.gdn_prepare(d["mixed_qkv"], d["conv_weight"], d["a_raw"], d["b_raw"], d["A_log"],
                  d["dt_bias"], d["cu_seqlens"], d["conv_pool"], q, k, v, g, beta, Hk=w.Hk,
                  Hv=w.Hv, Dk=w.Dk, Dv=w.Dv, K=w.K, state_indices=d["state_indices"],
                  has_initial_state=d["has_initial_state"],
                  cu_seqlens_host=w.cu_seqlens if host_mirrors else None,
                  state_indices_host=w.state_indices if host_mirrors else None,
                  apply_qk_l2norm=norm)
    return dict(q=q, k=k, v=v, g=g, beta=beta)


# ---- oracle ----------------------------------------------------------------------

def oracle_prepare(w: Workload, norm=True, nthreads=0):
    """O1 on the workload; returns the outputs and the updated conv pool (f32)."""
    pool = w.conv_pool.numpy().astype(np.float32).copy()
    out = oracle.prepare_varlen(
        f32(w.mixed_qkv), w.conv_weight.numpy(), pool, f32(w.a_raw), f32(w.b_raw),
        w.A_log.numpy(), w.dt_bias.numpy(), w.cu_seqlens.numpy(), w.Hk, w.Hv, w.Dk, w.Dv, w.K,
        state_indices=w.state_indices.numpy(), has_initial_state=w.has_initial_state.numpy(),
        apply_qk_l2norm=norm, dtype=np.float32, nthreads=nthreads)
    return out, pool


def compact_pool(w: Workload, seqs):
    """Initial states of the given sequences gathered into a compact f32 pool,
    and state indices that map those sequences to it (others -> -1)."""
    slots = [int(w.state_indices[s]) for s in seqs]
    live = [sl for sl in slots if sl >= 0]
    pool = np.zeros((max(len(live), 1), w.Hv, w.Dv, w.Dk), np.float32)
    remap = np.full(w.N, -1, np.int32)
    j = 0
    for s, sl in zip(seqs, slots):
        if sl >= 0:
            pool[j] = w.state_pool[sl].numpy()
            remap[s] = j
            j += 1
    return pool, remap


def seq_head_items(w: Workload, seqs, heads):
    return np.array([s * w.Hv + h for s in seqs for h in heads], np.int32)
