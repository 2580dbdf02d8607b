"""GPU parity of gdn_gated_rmsnorm against the oracle's gated RMSNorm
([cpu.rs] gated_rms_norm_f32; [cpu_ops.cpp] RmsNormGatedKernel's sigmoid gate
and strided gate rows), through the C ABI.  Inputs are seeded; bf16 outputs use
the bf16-storage metric of tests/helpers.py, f32 outputs the plain one."""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
from gated_delta_rule_44_gb300 import binding as B

pytestmark = pytest.mark.gpu


def run(T, Hh, D, dtype, sigmoid_gate, pad, dev, seed, eps=1e-6):
    g = torch.Generator().manual_seed(seed)
    core = (torch.randn(T, Hh, D, generator=g) * 3.0).to(dtype)
    zw = torch.randn(T, Hh * D + pad, generator=g).to(dtype)   # gate rows, padded
    w = (torch.rand(D, generator=g) + 0.5).to(dtype)
    out = torch.empty(T, Hh, D, dtype=dtype, device=dev)
    zd = zw.to(dev)
    B.gdn_gated_rmsnorm(core.to(dev), zd if pad else zd.view(T, Hh, D), w.to(dev), out, eps=eps,
                        sigmoid_gate=sigmoid_gate)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(H.f32(core), H.f32(zw), H.f32(w), eps, sigmoid_gate=sigmoid_gate,
                               dtype=np.float32)
    tol = H.TOL_F32 if dtype == torch.float32 else H.TOL_BF16
    return H.check(out, ref, tol, "gated_rmsnorm out")


@pytest.mark.parametrize("T,Hh,D,dtype,sig,pad", [
    (37, 3, 128, torch.bfloat16, False, 0),
    (64, 8, 64, torch.float32, True, 0),
    (17, 5, 128, torch.bfloat16, False, 24),     # gate rows of a wider projection
    (9, 2, 8, torch.bfloat16, True, 8),
    (5, 4, 1024, torch.bfloat16, False, 0),      # largest bf16 dim
    (6, 3, 512, torch.float32, False, 4),        # largest f32 dim
    (3, 7, 24, torch.bfloat16, False, 0),        # 3 vectors per row: group of 4 lanes, 1 idle
])
def test_gated_rmsnorm_matches_oracle(T, Hh, D, dtype, sig, pad, cuda_device):
    run(T, Hh, D, dtype, sig, pad, cuda_device, seed=T * 1000 + D)


def test_gated_rmsnorm_full_size(cuda_device):
    """The mixed workload's output shape: 8704 tokens x 64 value heads x 128."""
    e = run(8704, 64, 128, torch.bfloat16, False, 0, cuda_device, seed=5)
    print(f"gated_rmsnorm 8704x64x128: excess/rms {e:.2e}")


def test_gated_rmsnorm_eps_dominates(cuda_device):
    """A tiny row: eps sets the scale (1/sqrt(eps)), as in the closed form."""
    run(4, 2, 128, torch.float32, False, 0, cuda_device, seed=9, eps=1.0)
