"""Canary tails: every buffer a call writes is a view into a larger allocation
whose guard elements before and after it hold a NaN bit pattern; after the
call (and its device-status check) the guards must be bit-identical.  Covers
every entry point that writes device memory, on ragged shapes: the prepare
(q, k, v, g, beta and the conv pool), decode, the three prefill forms with
their workspace, the no-allocation prefill, KDA (recurrent and chunked, with
its workspace), speculative prepare and decode, packed decode, and the gated
RMSNorm.  A write past either end of any buffer fails here even when the
values it computes are right.

Also GDN_DEBUG_CHECKS=1: metadata passed in device memory only is copied to
the host and checked there, so a malformed cu_seqlens is refused before any
launch (in a child process, since the variable is read once)."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gated_delta_rule_44_gb300 import binding as B
from gated_delta_rule_44_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 1024  # elements before and after each buffer (2-4 KB: alignment is kept)
_PATTERN = {torch.bfloat16: (torch.int16, 0x7FC5), torch.float32: (torch.int32, 0x7FC0DEAD),
            torch.uint8: (torch.uint8, 0xA5)}


class Guarded:
    """A device buffer of `shape` with guard elements on both sides."""

    def __init__(self, shape, dtype, dev, init=None):
        n = int(np.prod(shape)) if len(shape) else 1
        idt, pat = _PATTERN[dtype]
        self.base = torch.empty(n + 2 * GUARD, dtype=dtype, device=dev)
        self.base.view(idt).fill_(pat if idt != torch.int16 else pat - 0x10000 * (pat > 0x7FFF))
        self.n, self.idt, self.pat = n, idt, pat
        self.t = self.base[GUARD:GUARD + n].view(shape)
        if init is not None:
            self.t.copy_(init)

    def check(self, what):
        torch.cuda.synchronize()
        g = torch.cat([self.base[:GUARD], self.base[GUARD + self.n:]]).view(self.idt)
        assert bool((g == self.pat).all()), f"{what}: a guard element was overwritten"


def workload(dev):
    w = W.make_workload("canary", 21, [1, 1, 1, 70, 129, 5], 2, 4, 128, 128, slots=9,
                        n_decode=3, state_std=0.1)
    d = dict(x=w.mixed_qkv.to(dev), w=w.conv_weight.to(dev), a=w.a_raw.to(dev),
             b=w.b_raw.to(dev), A_log=w.A_log.to(dev), dt_bias=w.dt_bias.to(dev),
             cu=w.cu_seqlens.to(dev), sidx=w.state_indices.to(dev),
             hinit=w.has_initial_state.to(dev))
    return w, d


def prepare(w, d, dev):
    outs = dict(q=Guarded((w.T, w.Hk, w.Dk), w.act_dtype, dev),
                k=Guarded((w.T, w.Hk, w.Dk), w.act_dtype, dev),
                v=Guarded((w.T, w.Hv, w.Dv), w.act_dtype, dev),
                g=Guarded((w.T, w.Hv), torch.float32, dev),
                beta=Guarded((w.T, w.Hv), torch.float32, dev),
                conv=Guarded(tuple(w.conv_pool.shape), torch.float32, dev, w.conv_pool))
    B.gdn_prepare(d["x"], d["w"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu"],
                  outs["conv"].t, outs["q"].t, outs["k"].t, outs["v"].t, outs["g"].t,
                  outs["beta"].t, Hk=w.Hk, Hv=w.Hv, Dk=w.Dk, Dv=w.Dv, K=w.K,
                  state_indices=d["sidx"], has_initial_state=d["hinit"])
    B.gdn_read_device_status()
    for k_, gb in outs.items():
        gb.check("prepare " + k_)
    return {k_: gb.t for k_, gb in outs.items()}


def test_prepare_decode_prefill_canaries(cuda_device):
    dev = cuda_device
    w, d = workload(dev)
    p = prepare(w, d, dev)
    nd = w.n_decode
    # decode rows, both output-norm placements included
    for norm in (None, "after", "in_kernel"):
        pool = Guarded(tuple(w.state_pool.shape), torch.float32, dev, w.state_pool)
        out = Guarded((nd, w.Hv, w.Dv), w.act_dtype, dev)
        kw = {}
        if norm is not None:
            kw = dict(norm_z=torch.randn(nd, w.Hv * w.Dv, device=dev).to(w.act_dtype),
                      norm_weight=torch.ones(w.Dv, device=dev, dtype=w.act_dtype),
                      norm_in_kernel=norm == "in_kernel")
        B.gdn_decode(p["q"][:nd], p["k"][:nd], p["v"][:nd], p["g"][:nd], p["beta"][:nd],
                     pool.t, out.t, state_indices=d["sidx"][:nd], **kw)
        B.gdn_read_device_status()
        pool.check(f"decode state ({norm})")
        out.check(f"decode out ({norm})")
    # the prefill rows on every form
    Tp, Np = w.T - nd, w.N - nd
    cup = (d["cu"][nd:] - nd).contiguous()
    for algo in (B.GDN_PREFILL_RECURRENT, B.GDN_PREFILL_CHUNKED, B.GDN_PREFILL_FUSED):
        pool = Guarded(tuple(w.state_pool.shape), torch.float32, dev, w.state_pool)
        out = Guarded((Tp, w.Hv, w.Dv), w.act_dtype, dev)
        nb = B.gdn_prefill_workspace_bytes(Tp, Np, w.Hv, w.Dk, w.Dv, 1, algo)
        ws = Guarded((nb,), torch.uint8, dev) if nb else None
        B.gdn_prefill_varlen(p["q"][nd:], p["k"][nd:], p["v"][nd:], p["g"][nd:],
                             p["beta"][nd:], pool.t, cup, out.t, state_indices=d["sidx"][nd:],
                             has_initial_state=d["hinit"][nd:], algo=algo,
                             workspace=None if ws is None else ws.t)
        B.gdn_read_device_status()
        pool.check(f"prefill state (algo {algo})")
        out.check(f"prefill out (algo {algo})")
        if ws is not None:
            ws.check(f"prefill workspace (algo {algo})")
    # the no-allocation entry point
    pool = Guarded(tuple(w.state_pool.shape), torch.float32, dev, w.state_pool)
    out = Guarded((Tp, w.Hv, w.Dv), w.act_dtype, dev)
    L = B.lib()
    fn = L.gdn_prefill_varlen_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(B.gdn_prefill_args), ctypes.c_void_p]
    qv, kv, vv, gv, bv = (p[n_][nd:] for n_ in ("q", "k", "v", "g", "beta"))
    args = B.gdn_prefill_args(
        T=Tp, N=Np, Hk=w.Hk, Hv=w.Hv, Dk=w.Dk, Dv=w.Dv, act_dtype=B.GDN_DTYPE_BF16,
        use_qk_l2norm=0, scale=-1.0, algo=B.GDN_PREFILL_CHUNKED, q=qv.data_ptr(), q_len=qv.numel(),
        k=kv.data_ptr(), k_len=kv.numel(), v=vv.data_ptr(), v_len=vv.numel(), g=gv.data_ptr(),
        g_len=gv.numel(), beta=bv.data_ptr(), beta_len=bv.numel(), state=pool.t.data_ptr(),
        state_slots=pool.t.shape[0], state_len=pool.t.numel(), cu_seqlens=cup.data_ptr(),
        state_indices=d["sidx"][nd:].data_ptr(), has_initial_state=d["hinit"][nd:].data_ptr(),
        cu_seqlens_host=None, state_indices_host=None, out=out.t.data_ptr(), out_len=out.t.numel(),
        workspace=None, workspace_bytes=0)
    assert fn(ctypes.byref(args), None) == B.GDN_OK, L.gdn_last_error_message()
    B.gdn_read_device_status()
    pool.check("noalloc prefill state")
    out.check("noalloc prefill out")
    # the gated RMSNorm
    out = Guarded((w.T, w.Hv, w.Dv), w.act_dtype, dev)
    B.gdn_gated_rmsnorm(p["v"], torch.randn(w.T, w.Hv, w.Dv, device=dev).to(w.act_dtype),
                        torch.ones(w.Dv, device=dev, dtype=w.act_dtype), out.t)
    out.check("gated rmsnorm out")


@pytest.mark.parametrize("algo", [B.GDN_PREFILL_RECURRENT, B.GDN_PREFILL_CHUNKED])
def test_kda_canaries(algo, cuda_device):
    dev = cuda_device
    g0 = torch.Generator().manual_seed(31)
    lens = [64, 1, 130, 7]
    T, N, Hk, Hv, D = sum(lens), len(lens), 2, 4, 128
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    q = (torch.randn(T, Hk, D, generator=g0) / D ** 0.5).to(torch.bfloat16).to(dev)
    k = (torch.randn(T, Hk, D, generator=g0) / D ** 0.5).to(torch.bfloat16).to(dev)
    v = torch.randn(T, Hv, D, generator=g0).to(torch.bfloat16).to(dev)
    g = (-torch.rand(T, Hv, D, generator=g0) * 0.3).to(dev)
    beta = torch.rand(T, Hv, generator=g0).to(dev)
    pool = Guarded((N + 2, Hv, D, D), torch.float32, dev, torch.randn(N + 2, Hv, D, D) * 0.1)
    out = Guarded((T, Hv, D), torch.bfloat16, dev)
    nb = B.gdn_kda_workspace_bytes(T, N, Hv, D, D, 1, algo)
    ws = Guarded((nb,), torch.uint8, dev) if nb else None
    B.gdn_kda_varlen(q, k, v, g, beta, pool.t, cu, out.t,
                     state_indices=torch.tensor([3, -1, 0, 5], dtype=torch.int32, device=dev),
                     algo=algo, workspace=None if ws is None else ws.t)
    B.gdn_read_device_status()
    pool.check("kda state")
    out.check("kda out")
    if ws is not None:
        ws.check("kda workspace")


def test_speculative_and_packed_canaries(cuda_device):
    dev = cuda_device
    g0 = torch.Generator().manual_seed(41)
    Hk, Hv, D, K, cols = 2, 4, 128, 4, 3
    lens = [3, 1, 0, 2]
    n, T = len(lens), sum(lens)
    C = 2 * Hk * D + Hv * D
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    x = torch.randn(T, C, generator=g0).to(torch.bfloat16).to(dev)
    wconv = (torch.randn(C, K, generator=g0) * 0.25).to(dev)
    a = torch.randn(T, Hv, generator=g0).to(torch.bfloat16).to(dev)
    b = torch.randn(T, Hv, generator=g0).to(torch.bfloat16).to(dev)
    A_log = torch.rand(Hv, generator=g0).add(1.0).log().to(dev)
    dt_bias = torch.randn(Hv, generator=g0).to(dev)
    width = (K - 1) + (cols - 1)
    conv = Guarded((6, C, width), torch.float32, dev, torch.randn(6, C, width, generator=g0))
    cidx = torch.tensor([4, 0, 2, 5], dtype=torch.int32, device=dev)
    nat = torch.tensor([1, 3, 2, 1], dtype=torch.int32, device=dev)
    q = Guarded((T, Hk, D), torch.bfloat16, dev)
    k = Guarded((T, Hk, D), torch.bfloat16, dev)
    v = Guarded((T, Hv, D), torch.bfloat16, dev)
    gg = Guarded((T, Hv), torch.float32, dev)
    bb = Guarded((T, Hv), torch.float32, dev)
    B.gdn_spec_prepare(x, wconv, a, b, A_log, dt_bias, cu, conv.t, cidx, nat, q.t, k.t, v.t, gg.t,
                       bb.t, Hk=Hk, Hv=Hv, Dk=D, Dv=D, K=K)
    B.gdn_read_device_status()
    for name, gb in dict(conv=conv, q=q, k=k, v=v, g=gg, beta=bb).items():
        gb.check("spec prepare " + name)
    slots = n * cols + 2
    pool = Guarded((slots, Hv, D, D), torch.float32, dev,
                   torch.randn(slots, Hv, D, D, generator=g0) * 0.1)
    sidx = torch.randperm(slots, generator=g0)[:n * cols].reshape(n, cols).to(torch.int32).to(dev)
    out = Guarded((T, Hv, D), torch.bfloat16, dev)
    B.gdn_spec_decode(q.t, k.t, v.t, gg.t, bb.t, pool.t, cu, sidx, nat, out.t)
    B.gdn_read_device_status()
    pool.check("spec decode state")
    out.check("spec decode out")
    # packed decode: one token per row
    Bn = 5
    xr = torch.randn(Bn, C, generator=g0).to(torch.bfloat16).to(dev)
    ar = torch.randn(Bn, Hv, generator=g0).to(torch.bfloat16).to(dev)
    br = torch.randn(Bn, Hv, generator=g0).to(torch.bfloat16).to(dev)
    pconv = Guarded((7, C, K - 1), torch.float32, dev, torch.randn(7, C, K - 1, generator=g0))
    pstate = Guarded((7, Hv, D, D), torch.float32, dev, torch.randn(7, Hv, D, D, generator=g0) * 0.1)
    pout = Guarded((Bn, Hv, D), torch.bfloat16, dev)
    pidx = torch.tensor([6, -1, 0, 3, 2], dtype=torch.int32, device=dev)
    B.gdn_packed_decode(xr, wconv, ar, br, A_log, dt_bias, pidx, pconv.t, pstate.t, pout.t,
                        Hk=Hk, Hv=Hv, Dk=D, Dv=D, K=K)
    B.gdn_read_device_status()
    pconv.check("packed decode conv")
    pstate.check("packed decode state")
    pout.check("packed decode out")


_DEBUG_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from gated_delta_rule_44_gb300 import binding as B
dev = torch.device("cuda:0")
T, N, Hk, Hv, D = 8, 2, 1, 2, 128
q = torch.randn(T, Hk, D, device=dev).to(torch.bfloat16)
v = torch.randn(T, Hv, D, device=dev).to(torch.bfloat16)
g = -torch.rand(T, Hv, device=dev)
beta = torch.rand(T, Hv, device=dev)
pool = torch.zeros(N, Hv, D, D, device=dev)
out = torch.empty(T, Hv, D, dtype=torch.bfloat16, device=dev)
cu = torch.tensor([0, 9, 8], dtype=torch.int32, device=dev)   # device only, malformed
try:
    B.gdn_prefill_varlen(q, q, v, g, beta, pool, cu, out, algo=B.GDN_PREFILL_RECURRENT)
    B.gdn_read_device_status()
    print("RESULT ok")
except B.GdnError as e:
    print("RESULT", e.code, e.msg)
"""


@pytest.mark.parametrize("debug", [False, True])
def test_debug_checks_refuse_device_only_metadata(debug, cuda_device):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    env.pop("GDN_DEBUG_CHECKS", None)
    if debug:
        env["GDN_DEBUG_CHECKS"] = "1"
    r = subprocess.run([sys.executable, "-c", _DEBUG_CHILD, root], env=env, capture_output=True,
                       text=True, timeout=600)
    line = [x for x in r.stdout.splitlines() if x.startswith("RESULT")]
    assert r.returncode == 0 and line, r.stdout + r.stderr
    if debug:  # refused on the host, before any launch, with the page's message
        assert line[0] == ("RESULT 2 gated_delta_rule_varlen sequence 1 has empty or "
                           "non-monotonic range 9..8"), line[0]
    else:      # launched; the kernel's own check reports it through the status word
        assert line[0].startswith(f"RESULT {B.GDN_ERR_DEVICE_CHECK}"), line[0]
