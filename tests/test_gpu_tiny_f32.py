"""The tiny f32 workload end to end on the GPU, on its own seeded inputs.

One 64-token sequence, Hk=2, Hv=4, Dk=Dv=32, conv width 4, f32 activations and
a zero initial state (seed 0): gdn_prepare (conv1d + SiLU + split + q/k L2 norm
+ gates, [cpu.rs] linear_attention_prepare_varlen_f32) then gdn_prefill_varlen
([cpu.rs] recurrent_gated_delta_rule_varlen_f32), both through the C ABI,
against the oracle's prepare (O1) and recurrence (O2) on the same raw inputs,
at the f32 tolerance max|err|/rms(ref) <= 1e-4 for every output of both steps,
the final state and the conv tail.  Nothing is rounded between the steps: the
path stores f32.  Its weak-decay twin runs the same way.
"""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B
from gated_delta_rule_44_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("weak", [False, True])
@pytest.mark.parametrize("algo", [B.GDN_PREFILL_AUTO, B.GDN_PREFILL_RECURRENT])
def test_tiny_f32_end_to_end(weak, algo, cuda_device):
    dev = cuda_device
    w = W.named("tiny_f32", weak_decay=weak)
    assert w.act_dtype == torch.float32 and w.T == 64 and w.N == 1
    d = H.to_dev(w, dev)
    got = H.gpu_prepare(w, d)
    out = torch.full((w.T, w.Hv, w.Dv), float("nan"), device=dev)
    B.gdn_prefill_varlen(got["q"], got["k"], got["v"], got["g"], got["beta"], d["state_pool"],
                         d["cu_seqlens"], out, state_indices=d["state_indices"],
                         has_initial_state=d["has_initial_state"],
                         cu_seqlens_host=w.cu_seqlens, state_indices_host=w.state_indices,
                         algo=algo)
    B.gdn_read_device_status()

    ref_prep, ref_conv = H.oracle_prepare(w)
    for key in ("q", "k", "v", "g", "beta"):
        H.check(got[key], ref_prep[key], H.TOL_F32, key)
    np.testing.assert_array_equal(H.f32(d["conv_pool"]), ref_conv)
    pool = w.state_pool.numpy().copy()
    ref_out = oracle.gdn_varlen(ref_prep["q"], ref_prep["k"], ref_prep["v"], ref_prep["g"],
                                ref_prep["beta"], pool, w.cu_seqlens.numpy(),
                                1.0 / np.sqrt(w.Dk), state_indices=w.state_indices.numpy(),
                                has_initial_state=w.has_initial_state.numpy(), dtype=np.float32)
    e_out = H.check(out, ref_out, H.TOL_F32, "out")
    e_state = H.assert_close(H.f32(d["state_pool"]), pool, H.TOL_F32, "state")
    print(f"tiny_f32 weak={weak}: out err {e_out:.2e}, state err {e_state:.2e}")
