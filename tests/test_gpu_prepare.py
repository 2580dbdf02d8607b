"""GPU parity of gdn_prepare against the oracle's prepare step (O1).

Small cases span several token tiles and channel blocks, ragged sequence
lengths (1, 2, 3, K-1, K, 63, 64, 65, ...), padding slots (-1), a mix of
has_initial_state, conv widths 2..6, f32 and bf16, and more than 1024
sequences; the five named workloads run at full size.  q, k, v, g, beta must match within the parity tolerance (q, k, v with the
bf16-storage metric of tests/helpers.py when stored in bf16); the conv-tail
pool holds raw inputs and must match bit for bit.
"""
import numpy as np
import pytest
import torch

import helpers as H
from gated_delta_rule_44_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def check(w, dev, norm=True, host_mirrors=True):
    d = H.to_dev(w, dev)
    got = H.gpu_prepare(w, d, norm=norm, host_mirrors=host_mirrors)
    ref, ref_pool = H.oracle_prepare(w, norm=norm)
    tol = H.tol_for(w)
    errs = {}
    for key in ("q", "k", "v", "g", "beta"):
        errs[key] = H.check(got[key], ref[key], tol, key)
    np.testing.assert_array_equal(H.f32(d["conv_pool"]), ref_pool)
    return errs


CASES = [
    # seqlens, Hk, Hv, Dk, Dv, K, dtype, padded, prefill_new
    ([64], 2, 4, 32, 32, 4, torch.float32, None, False),
    ([1, 2, 3, 4, 5, 63, 64, 65, 130, 7], 2, 4, 32, 32, 4, torch.bfloat16, None, False),
    ([1, 2, 3, 4, 5, 63, 64, 65, 130, 7], 2, 4, 32, 16, 4, torch.float32, [2, 6], False),
    ([3, 17, 1, 1, 1, 40], 2, 6, 64, 64, 2, torch.bfloat16, [3], True),
    ([3, 17, 1, 1, 1, 40], 1, 2, 16, 24, 3, torch.bfloat16, None, False),
    ([9, 300, 2], 4, 8, 128, 128, 4, torch.bfloat16, None, False),
    ([5, 33], 2, 2, 8, 8, 6, torch.float32, None, False),
    ([1] * 37, 2, 4, 256, 64, 4, torch.bfloat16, [0, 36], False),
    # more than 1024 sequences: the tile's sequence search takes three rounds;
    # one-token rows around longer sequences, with padding slots
    ([1] * 1030 + [70, 3, 130] + [1] * 40, 1, 2, 16, 16, 4, torch.bfloat16, [5, 1031], False),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prepare_small(case, cuda_device):
    seqlens, Hk, Hv, Dk, Dv, K, dt, padded, new = CASES[case]
    w = W.make_workload("t", 100 + case, seqlens, Hk, Hv, Dk, Dv, K=K, act_dtype=dt,
                        slots=len(seqlens) + 3, padded=padded, prefill_new=new, n_decode=1)
    check(w, cuda_device)


def test_prepare_without_norm_and_mirrors(cuda_device):
    w = W.make_workload("t", 7, [5, 70, 2], 2, 4, 32, 32, act_dtype=torch.bfloat16)
    check(w, cuda_device, norm=False, host_mirrors=False)


def test_prepare_strided_rows(cuda_device):
    # mixed_qkv and a/b as views into wider rows
    w = W.make_workload("t", 8, [20, 11], 2, 4, 32, 32, act_dtype=torch.bfloat16)
    d = H.to_dev(w, cuda_device)
    C = w.C_conv
    wide = torch.zeros((w.T, C + 24), dtype=w.act_dtype, device=cuda_device)
    wide[:, 8:8 + C] = d["mixed_qkv"]
    d["mixed_qkv"] = wide[:, 8:8 + C]
    ab = torch.zeros((w.T, 2 * w.Hv + 3), dtype=w.act_dtype, device=cuda_device)
    ab[:, :w.Hv] = d["b_raw"]
    ab[:, w.Hv + 3:] = d["a_raw"]
    d["b_raw"], d["a_raw"] = ab[:, :w.Hv], ab[:, w.Hv + 3:]
    got = H.gpu_prepare(w, d)
    ref, ref_pool = H.oracle_prepare(w)
    for key in ("q", "k", "v", "g", "beta"):
        H.check(got[key], ref[key], H.tol_for(w), key)
    np.testing.assert_array_equal(H.f32(d["conv_pool"]), ref_pool)


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_prepare_named_full_size(name, cuda_device):
    check(W.named(name), cuda_device)
