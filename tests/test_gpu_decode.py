"""GPU parity of gdn_decode against the oracle's decode (O3).

Inputs: the oracle's own prepare outputs, rounded to the activation dtype by
torch; the oracle then receives exactly those rounded values (widened), so both
sides see identical inputs.  Covers Dk in {16, 32, 64, 128, 256}, ragged Dv,
GQA ratios, padding rows (-1), NULL indices, in-kernel q/k norm, an explicit
scale, f32 and bf16, the decode workload at full size and its weak-decay twin.
The output and the whole state pool are compared (untouched slots exactly).
"""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B
from gated_delta_rule_44_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_decode(w, dev, scale=-1.0, null_indices=False, norm=False, host_mirror=True):
    ref_prep, _ = H.oracle_prepare(w, norm=not norm)
    acts = {k: torch.from_numpy(ref_prep[k]).to(w.act_dtype) for k in ("q", "k", "v")}
    g = torch.from_numpy(ref_prep["g"])
    beta = torch.from_numpy(ref_prep["beta"])
    sidx = None if null_indices else w.state_indices
    out = torch.empty((w.T, w.Hv, w.Dv), dtype=w.act_dtype, device=dev)
    pool = w.state_pool.to(dev)
    B.gdn_decode(acts["q"].to(dev), acts["k"].to(dev), acts["v"].to(dev), g.to(dev),
                 beta.to(dev), pool, out, scale=scale,
                 state_indices=None if sidx is None else sidx.to(dev),
                 state_indices_host=sidx if host_mirror else None, use_qk_l2norm=norm)
    B.gdn_read_device_status()
    ref_pool = w.state_pool.numpy().copy()
    sc = scale if scale >= 0 else 1.0 / np.sqrt(w.Dk)
    ref_out = oracle.gdn_decode(H.f32(acts["q"]), H.f32(acts["k"]), H.f32(acts["v"]),
                                g.numpy(), beta.numpy(), ref_pool, sc,
                                state_indices=None if sidx is None else sidx.numpy(),
                                use_qk_l2norm=norm, dtype=np.float32)
    tol = H.tol_for(w)
    e_out = H.check(out, ref_out, tol, "out")
    got_pool = H.f32(pool)
    live = sorted({int(s) for s in (sidx.tolist() if sidx is not None else range(w.T)) if s >= 0})
    e_state = H.assert_close(got_pool[live], ref_pool[live], tol, "state")
    dead = [s for s in range(w.slots) if s not in set(live)]
    np.testing.assert_array_equal(got_pool[dead], ref_pool[dead])
    return e_out, e_state


CASES = [
    # B, Hk, Hv, Dk, Dv, dtype, padded
    (5, 2, 4, 32, 32, torch.float32, None),
    (7, 1, 3, 16, 40, torch.float32, [1]),
    (9, 2, 8, 64, 64, torch.bfloat16, [0, 8]),
    (33, 4, 8, 128, 128, torch.bfloat16, [5]),
    (6, 2, 2, 128, 72, torch.float32, None),
    (4, 1, 2, 256, 128, torch.bfloat16, None),
    (3, 2, 4, 256, 256, torch.float32, [2]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_small(case, cuda_device):
    Bn, Hk, Hv, Dk, Dv, dt, padded = CASES[case]
    w = W.make_workload("d", 200 + case, [1] * Bn, Hk, Hv, Dk, Dv, act_dtype=dt, slots=Bn + 5,
                        padded=padded, n_decode=Bn, state_std=0.3)
    run_decode(w, cuda_device)


def test_decode_null_indices_norm_and_scale(cuda_device):
    w = W.make_workload("d", 210, [1] * 12, 2, 4, 128, 128, act_dtype=torch.bfloat16,
                        permute_slots=False, n_decode=12, state_std=0.3)
    run_decode(w, cuda_device, null_indices=True)
    run_decode(w, cuda_device, norm=True, scale=0.37)
    run_decode(w, cuda_device, host_mirror=False)


@pytest.mark.parametrize("weak", [False, True])
def test_decode_b256_full_size(weak, cuda_device):
    w = W.named("decode_b256", weak_decay=weak)
    e_out, e_state = run_decode(w, cuda_device)
    print(f"decode_b256 weak={weak}: out err {e_out:.2e}, state err {e_state:.2e}")
