"""GPU parity of the output-norm option of gdn_decode and gdn_prefill_varlen:
the gated RMSNorm ([cpu.rs] gated_rms_norm_f32; [cpu_ops.cpp]
RmsNormGatedKernel) applied where the recurrence stores its output
([qwen3_5.cpp] the gated output norm after the attention core).

Expected values: the oracle's recurrence (O2 / O3) on the same seeded inputs,
its output rounded to the activation type as the unfused pipeline stores it,
then the oracle's gated RMSNorm.  The comparison allows, per element, the
recurrence's own tolerance carried through the norm (a core error of tol *
rms(core) moves an output by at most that times |out / core| of the row:
inv_rms * |weight * gate|), on top of the storage metric of tests/helpers.py.
Also: the state a normed call leaves equals the state of the plain call bit
for bit, and the normed output agrees with the standalone norm kernel run on
the plain call's output (GPU against GPU) to one bf16 step (bit for bit where
the call runs that kernel itself).  The decode is checked on both routes: the
norm kernel after the recurrence (the default) and inside the decode kernel.
"""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B
from gated_delta_rule_44_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def gate_inputs(T, Hv, Dv, dtype, pad, seed):
    g = torch.Generator().manual_seed(seed)
    zw = torch.randn(T, Hv * Dv + pad, generator=g).to(dtype)  # gate rows, maybe padded
    w = (torch.rand(Dv, generator=g) + 0.5).to(dtype)
    return zw, w


def expected(core_ref, zw, w, eps, sig, act_dtype):
    """The oracle's norm of the stored core, and the per-element allowance."""
    core_ref = np.asarray(core_ref, dtype=np.float64)
    stored = H.bf16_round(core_ref) if act_dtype == torch.bfloat16 else core_ref.astype(
        np.float32).astype(np.float64)
    ref = oracle.gated_rmsnorm(stored, H.f32(zw).astype(np.float64),
                               H.f32(w).astype(np.float64), eps, sigmoid_gate=sig)
    # |out / core| is the same for every element of a row whose core is not
    # zero; for a row of zeros it does not matter (the output is zero)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(stored != 0, np.abs(ref / np.where(stored != 0, stored, 1.0)), 0.0)
    tol = H.TOL_F32 if act_dtype == torch.float32 else H.TOL_BF16
    rms_core = float(np.sqrt((core_ref ** 2).mean())) or 1.0
    return ref, tol * rms_core * ratio, tol


def compare(out_norm, out_plain, core_ref, zw, w, eps, sig, act_dtype, dev, what):
    T, Hv, Dv = out_norm.shape
    ref, extra, tol = expected(core_ref, zw, w, eps, sig, act_dtype)
    got = H.f32(out_norm).astype(np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    H.assert_close(got, ref, tol, f"{what} vs oracle", stored_bf16=act_dtype == torch.bfloat16,
                   extra=extra)
    # GPU against GPU: the standalone norm of the plain output
    zd = zw.to(dev)
    sep = torch.empty_like(out_plain)
    B.gdn_gated_rmsnorm(out_plain, zd, w.to(dev), sep, eps=eps, sigmoid_gate=sig)
    torch.cuda.synchronize()
    a, b = H.f32(out_norm).astype(np.float64), H.f32(sep).astype(np.float64)
    step = H.bf16_quantum(b) if act_dtype == torch.bfloat16 else 1e-5 * np.abs(b) + 1e-30
    assert np.all(np.abs(a - b) <= step + 1e-30), f"{what}: fused and standalone norms differ"


def run_decode_case(Bn, Hk, Hv, Dk, Dv, dtype, padded, sig, pad, dev, seed, in_kernel=False):
    w = W.make_workload("d", seed, [1] * Bn, Hk, Hv, Dk, Dv, act_dtype=dtype, slots=Bn + 3,
                        padded=padded, n_decode=Bn, state_std=0.3)
    prep, _ = H.oracle_prepare(w)
    acts = {k: torch.from_numpy(prep[k]).to(dtype) for k in ("q", "k", "v")}
    g, beta = torch.from_numpy(prep["g"]), torch.from_numpy(prep["beta"])
    zw, wt = gate_inputs(Bn, Hv, Dv, dtype, pad, seed)
    eps = 1e-6
    outs, pools = [], []
    for normed in (False, True):
        pool = w.state_pool.to(dev)
        out = torch.full((Bn, Hv, Dv), 7.0, dtype=dtype, device=dev)
        zd = zw.to(dev)
        B.gdn_decode(acts["q"].to(dev), acts["k"].to(dev), acts["v"].to(dev), g.to(dev),
                     beta.to(dev), pool, out, state_indices=w.state_indices.to(dev),
                     norm_z=zd if normed else None, norm_weight=wt.to(dev) if normed else None,
                     norm_eps=eps, norm_sigmoid=sig, norm_in_kernel=in_kernel)
        B.gdn_read_device_status()
        outs.append(out)
        pools.append(pool)
    assert torch.equal(pools[0], pools[1]), "the norm changed the state"
    ref_pool = w.state_pool.numpy().astype(np.float64)
    core_ref = oracle.gdn_decode(H.f32(acts["q"]), H.f32(acts["k"]), H.f32(acts["v"]),
                                 g.numpy(), beta.numpy(), ref_pool, 1.0 / np.sqrt(Dk),
                                 state_indices=w.state_indices.numpy(), dtype=np.float64)
    compare(outs[1], outs[0], core_ref, zw, wt, eps, sig, dtype, dev,
            f"decode B{Bn} Dk{Dk} Dv{Dv}" + (" in kernel" if in_kernel else ""))
    if padded:  # padding rows stay zero
        assert torch.all(outs[1][padded].float() == 0)


DECODE_CASES = [
    # B, Hk, Hv, Dk, Dv, dtype, padded rows, sigmoid gate, gate-row padding
    (9, 2, 4, 128, 128, torch.bfloat16, [3], False, 0),    # two slices in one CTA
    (5, 1, 2, 128, 256, torch.bfloat16, None, True, 16),   # four slices: the widest CTA
    (4, 1, 2, 256, 256, torch.bfloat16, None, False, 0),   # eight slices: the norm kernel after
    (6, 2, 2, 64, 64, torch.float32, [0], False, 4),       # one slice
    (3, 1, 3, 16, 1024, torch.bfloat16, None, False, 8),   # eight slices of 128 rows
    (3, 1, 2, 32, 256, torch.bfloat16, None, True, 0),     # four slices of 64 rows
    (7, 2, 2, 128, 96, torch.float32, None, True, 0),      # a ragged second slice
]


@pytest.mark.parametrize("in_kernel", [False, True])
@pytest.mark.parametrize("case", range(len(DECODE_CASES)))
def test_decode_out_norm(case, in_kernel, cuda_device):
    run_decode_case(*DECODE_CASES[case], cuda_device, seed=900 + case, in_kernel=in_kernel)


def run_prefill_case(lens, Hk, Hv, dtype, algo, sig, pad, dev, seed, Dk=128, Dv=128):
    w = W.make_workload("p", seed, lens, Hk, Hv, Dk, Dv, act_dtype=dtype, slots=len(lens) + 2,
                        state_std=0.3)
    prep, _ = H.oracle_prepare(w)
    acts = {k: torch.from_numpy(prep[k]).to(dtype) for k in ("q", "k", "v")}
    g, beta = torch.from_numpy(prep["g"]), torch.from_numpy(prep["beta"])
    T, N = w.T, w.N
    zw, wt = gate_inputs(T, Hv, Dv, dtype, pad, seed)
    eps = 1e-5
    nbytes = B.gdn_prefill_workspace_bytes(T, N, Hv, Dk, Dv, B._dt(acts["q"]), algo)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev) if nbytes else None
    outs, pools = [], []
    for normed in (False, True):
        pool = w.state_pool.to(dev)
        out = torch.full((T, Hv, Dv), 7.0, dtype=dtype, device=dev)
        B.gdn_prefill_varlen(acts["q"].to(dev), acts["k"].to(dev), acts["v"].to(dev), g.to(dev),
                             beta.to(dev), pool, w.cu_seqlens.to(dev), out,
                             state_indices=w.state_indices.to(dev),
                             has_initial_state=w.has_initial_state.to(dev), algo=algo,
                             workspace=ws, norm_z=zw.to(dev) if normed else None,
                             norm_weight=wt.to(dev) if normed else None, norm_eps=eps,
                             norm_sigmoid=sig)
        B.gdn_read_device_status()
        outs.append(out)
        pools.append(pool)
    assert torch.equal(pools[0], pools[1]), "the norm changed the state"
    ref_pool = w.state_pool.numpy().astype(np.float64)
    core_ref = oracle.gdn_varlen(H.f32(acts["q"]), H.f32(acts["k"]), H.f32(acts["v"]),
                                 g.numpy(), beta.numpy(), ref_pool, w.cu_seqlens.numpy(),
                                 1.0 / np.sqrt(Dk), state_indices=w.state_indices.numpy(),
                                 has_initial_state=w.has_initial_state.numpy(), dtype=np.float64)
    compare(outs[1], outs[0], core_ref, zw, wt, eps, sig, dtype, dev,
            f"prefill algo {algo} lens {lens}")


PREFILL_CASES = [
    # lens, Hk, Hv, dtype, algo, sigmoid gate, gate-row padding
    ([70, 1, 129], 2, 4, torch.bfloat16, B.GDN_PREFILL_FUSED, False, 0),
    ([64, 200], 1, 2, torch.bfloat16, B.GDN_PREFILL_FUSED, True, 8),
    ([70, 1, 129], 2, 4, torch.bfloat16, B.GDN_PREFILL_CHUNKED, False, 0),
    ([33, 5], 1, 2, torch.bfloat16, B.GDN_PREFILL_RECURRENT, True, 24),
    ([20, 9, 3], 1, 2, torch.float32, B.GDN_PREFILL_RECURRENT, False, 0),
]


@pytest.mark.parametrize("case", range(len(PREFILL_CASES)))
def test_prefill_out_norm(case, cuda_device):
    run_prefill_case(*PREFILL_CASES[case], cuda_device, seed=950 + case)
