"""Shared test helpers: run the CUDA path and the oracle on the same seeded
workload and compare them.

The parity metric is the one the layer is specified with:
    err = max |gpu - ref| / rms(ref)
over the whole compared tensor, with tolerance 1e-4 for f32 activations and
2e-2 for bf16 activations (state always f32).

Tensors the path STORES in bf16 (q, k, v, out) are compared the way the pages
store them: the pages' store rounds an f32 result to the storage type
(round-to-nearest-even; vllm.cpp cpu_ops.cpp StoreF32), so the reference is the
oracle's f32 result rounded to bf16.  When the GPU's and the oracle's f32 values
straddle a rounding boundary the two sides legitimately pick neighbouring bf16
values, so a difference of one bf16 quantum (the spacing at the reference
value) is exempt; every difference beyond it counts in full:
    err = max(|gpu - bf16(ref)| - quantum(bf16(ref)), 0) / rms(ref).
f32 tensors (state, g, beta) use the plain metric.  Every bf16 comparison also
reports and bounds rms(gpu - ref)/rms(ref), the plain metric averaged, so that
a systematic one-quantum bias cannot hide under the exemption.

End to end (prepare, then the recurrence, from raw inputs) the same holds one
step earlier: q, k and v are stored in bf16 between the two steps, and where
the path's and the oracle's f32 values straddle a rounding boundary the two
stored values differ by one step, which the recurrence carries into the
outputs (measured on the oracle alone: flipping the near-boundary q or k
values of a D = 128 head moves outputs by up to 3e-2 of their rms).
stored_flip_bound bounds this from the oracle's own values, with the
oracle's first-order deviation bound of the recurrence, and the end-to-end
tests add it to the exemption.

Oracle inputs come only from the workload generator (bf16 values widened
exactly to f32) or from the oracle's own earlier steps (rounded to bf16 where
the path stores bf16), never from the CUDA path.
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


def bf16_round(x) -> np.ndarray:
    """Round-to-nearest-even to bf16, returned as f64 (torch's conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def bf16_quantum(xq: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at each (bf16) value: 2^(exponent - 7); 0 at 0."""
    a = np.abs(np.asarray(xq, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def rel_err_stored_bf16(gpu, ref, extra=None) -> float:
    """max(|gpu - bf16(ref)| - one bf16 quantum - extra, 0) / rms(ref); `extra`
    (same shape, default 0) is a per-element allowance such as
    stored_flip_bound's."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rq = bf16_round(ref)
    excess = np.abs(gpu - rq) - bf16_quantum(rq)
    if extra is not None:
        excess -= np.asarray(extra, dtype=np.float64)
    excess = np.maximum(excess, 0.0)
    rms = float(np.sqrt((ref ** 2).mean()))
    return float(excess.max()) / rms if rms > 0 else float(excess.max())


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


def rms_rel_err(gpu, ref) -> float:
    """rms(gpu - ref) / rms(ref) over the whole tensor: a systematic bias of
    a bf16 quantum or so shows here even where the max metric exempts it."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt((ref ** 2).mean()))
    d = float(np.sqrt(((gpu - ref) ** 2).mean()))
    return d / rms if rms > 0 else d


def bf16_flip(x):
    """For each value x, its bf16 rounding r, the neighbouring bf16 value nb on
    the side of x, and |x - (r + nb) / 2|, its distance from the rounding
    boundary between them (computed on the bf16 bit patterns, so binade
    edges are exact).  Zeros and exact bf16 values get nb = r."""
    x = np.asarray(x, dtype=np.float64)
    r = bf16_round(x)
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.int64)
    up = x > r                       # x lies above its rounding
    away = np.where(r > 0, up, ~up)  # toward larger magnitude
    step = np.where(x == r, 0, np.where(away, 1, -1))
    step = np.where(r == 0, 0, step)
    nb = ((bits + step).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    dist = np.abs(x - 0.5 * (r + nb))
    return r, nb, dist


def stored_flip_bound(prep, cu_seqlens, scale, state_pool, state_indices=None,
                      has_initial_state=None, margin=1.0 / 32):
    """Allowance for outputs computed end to end from raw inputs, where q, k
    and v are stored in bf16 between the prepare and the recurrence by two
    different f32 evaluations of the same prepare (the path's and the
    oracle's).  Where the oracle's f32 value lies within `margin` of a bf16
    step of a rounding boundary, the other evaluation may store the
    neighbouring value; every other stored value is the same on both sides.
    Returns the oracle's first-order bound (oracle.gdn_deviation_bound) on
    how far those one-step moves can carry each output of the recurrence, and
    a bound on every element of each row of each live final state
    ([slots, Hv, Dv])."""
    rounded, moves = {}, {}
    for key in ("q", "k", "v"):
        r, nb, dist = bf16_flip(prep[key])
        step = np.abs(nb - r)
        rounded[key] = r
        moves[key] = np.where((step > 0) & (dist <= margin * step), step, 0.0)
    return oracle.gdn_deviation_bound(
        rounded["q"], rounded["k"], rounded["v"], prep["g"], prep["beta"], moves["q"],
        moves["k"], moves["v"], state_pool, cu_seqlens, scale, state_indices=state_indices,
        has_initial_state=has_initial_state, with_state=True)


def assert_close(gpu, ref, tol, what="", stored_bf16=False, extra=None):
    """Plain metric for f32 tensors; the storage-rounding metric (see the module
    docstring) for tensors the path stores in bf16, which must also keep
    rms(err)/rms(ref) within the tolerance.  `extra`: a per-element allowance
    added to the one-quantum exemption (stored_flip_bound).  Returns the
    error."""
    assert np.all(np.isfinite(np.asarray(gpu, dtype=np.float64))), f"{what}: non-finite"
    if stored_bf16:
        e = rel_err_stored_bf16(gpu, ref, extra)
        e_plain = rel_err(gpu, ref)
        e_rms = rms_rel_err(gpu, ref)
        print(f"{what}: max(|err| - 1 bf16 quantum)/rms(ref) {e:.3e}, plain max|err|/rms "
              f"{e_plain:.3e}, rms(err)/rms(ref) {e_rms:.3e}")
        assert e <= tol, (f"{what}: max(|err| - 1 bf16 quantum)/rms(ref) = {e:.3e} > {tol:.1e}"
                          f" (plain max|err|/rms = {e_plain:.3e})")
        assert e_rms <= tol, f"{what}: rms(err)/rms(ref) = {e_rms:.3e} > {tol:.1e}"
        return e
    e = rel_err(gpu, ref)
    assert e <= tol, f"{what}: max|err|/rms(ref) = {e:.3e} > {tol:.1e}"
    return e


def assert_close_blocks(pairs, tol, what=""):
    """The plain metric (max|err| / rms(ref)) over the concatenation of
    (gpu, ref[, extra]) array tuples, without materialising it: for large state
    pools.  `extra` (optional, broadcastable to the block) is a per-element
    allowance subtracted from |err| first (stored_flip_bound's state bound)."""
    mx, ss, n = 0.0, 0.0, 0
    for blk in pairs:
        gpu, ref = blk[0], blk[1]
        g = np.asarray(gpu, dtype=np.float64)
        r = np.asarray(ref, dtype=np.float64)
        assert g.shape == r.shape, (g.shape, r.shape)
        assert np.all(np.isfinite(g)), f"{what}: non-finite"
        if r.size:
            d = np.abs(g - r)
            if len(blk) > 2 and blk[2] is not None:
                d = np.maximum(d - np.asarray(blk[2], dtype=np.float64), 0.0)
            mx = max(mx, float(d.max()))
            ss += float((r * r).sum())
            n += r.size
    rms = np.sqrt(ss / n) if n else 0.0
    e = mx / rms if rms > 0 else mx
    assert e <= tol, f"{what}: max|err|/rms(ref) = {e:.3e} > {tol:.1e}"
    return e


def check(gpu_t: torch.Tensor, ref, tol, what=""):
    """assert_close with the metric chosen by the GPU tensor's storage dtype."""
    return assert_close(f32(gpu_t), ref, tol, what, stored_bf16=gpu_t.dtype == torch.bfloat16)


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
