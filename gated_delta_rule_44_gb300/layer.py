"""One GDN layer step over a packed batch: the three library calls in order.

Mixed batches follow [qwen3_5.cpp] (vllm.cpp, src/vllm/model_executor/models/
qwen3_5.cpp) ValidateGdnAttentionMetadata and SubView: the decode rows come
first (one token each), then the prefill sequences.  One ``gdn_prepare`` runs
over every token; ``gdn_decode`` then takes rows [0, n_decode) and
``gdn_prefill_varlen`` the rest, with its cu_seqlens rebased to start at 0
(the caller's ``cu_seqlens_prefill``, like the pages' prefill_query_start_loc).
All buffers are torch tensors on one device; everything is asynchronous on the
given stream.

``GdnHostPipeline`` serves callers whose per-step inputs and outputs live in
pinned host memory: it copies a step's inputs in and its output out on their
own streams, so that they overlap the neighbouring steps' compute; the steps'
compute stays in order on one stream (each step updates the state and conv
pools the next one reads).
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class GdnStep:
    """Preallocated intermediates (q, k, v, g, beta, out, prefill workspace) for
    batches of a fixed token count, and the three calls of one step."""

    def __init__(self, T: int, N: int, n_decode: int, Hk: int, Hv: int, Dk: int, Dv: int, K: int,
                 act_dtype: torch.dtype, device, scale: float = -1.0,
                 algo: int = B.GDN_PREFILL_AUTO, apply_qk_l2norm: bool = True):
        self.T, self.N, self.n_decode = T, N, n_decode
        self.Hk, self.Hv, self.Dk, self.Dv, self.K = Hk, Hv, Dk, Dv, K
        self.scale, self.algo, self.norm = scale, algo, apply_qk_l2norm
        dev = torch.device(device)
        self.q = torch.empty((T, Hk, Dk), dtype=act_dtype, device=dev)
        self.k = torch.empty((T, Hk, Dk), dtype=act_dtype, device=dev)
        self.v = torch.empty((T, Hv, Dv), dtype=act_dtype, device=dev)
        self.g = torch.empty((T, Hv), dtype=torch.float32, device=dev)
        self.beta = torch.empty((T, Hv), dtype=torch.float32, device=dev)
        self.out = torch.empty((T, Hv, Dv), dtype=act_dtype, device=dev)
        self.nd_tok = n_decode
        Tp, Np = T - self.nd_tok, N - n_decode
        dt = B.GDN_DTYPE_BF16 if act_dtype == torch.bfloat16 else B.GDN_DTYPE_F32
        ws = B.gdn_prefill_workspace_bytes(Tp, Np, Hv, Dk, Dv, dt, algo) if Np > 0 else 0
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev) if ws else None

    def validate(self, cu_seqlens_host, state_indices_host, cu_seqlens_prefill_host,
                 has_initial_state_host=None, state_slots=None) -> None:
        """Checks host copies of the step's metadata against the mixed-step
        contract ([qwen3_5.cpp] ValidateGdnAttentionMetadata, via the C ABI's
        gdn_validate_mixed): decode rows first and single-token,
        cu_seqlens[n_decode] == n_decode, the prefill cu_seqlens equal to the
        suffix of cu_seqlens rebased to 0, the prefill indices the suffix of
        state_indices.  Raises GdnError; launches nothing."""
        nd = self.n_decode
        if state_slots is None:
            state_slots = (int(state_indices_host.max().item()) + 1
                           if state_indices_host.numel() else 0)
        B.gdn_validate_mixed(num_decodes=nd, num_prefills=self.N - nd,
                             num_actual_tokens=self.T, state_slots=state_slots,
                             cu_seqlens_host=cu_seqlens_host,
                             state_indices_host=state_indices_host,
                             has_initial_state_host=has_initial_state_host,
                             cu_seqlens_prefill_host=(cu_seqlens_prefill_host
                                                      if self.N > nd else None))

    def run(self, mixed_qkv, a_raw, b_raw, conv_weight, A_log, dt_bias, cu_seqlens, state_indices,
            has_initial_state, state_pool, conv_pool, cu_seqlens_prefill=None,
            stream: Optional[torch.cuda.Stream] = None,
            out: Optional[torch.Tensor] = None, cu_seqlens_host=None, state_indices_host=None,
            has_initial_state_host=None, cu_seqlens_prefill_host=None) -> torch.Tensor:
        """One step; writes the output to ``out`` (default: this object's own
        buffer) and returns it.  When host copies of the metadata are passed
        (``*_host``), the step's metadata contract is checked before anything
        is launched (see ``validate``) and the calls get the host mirrors for
        their own index and cu_seqlens checks."""
        nd, ndt = self.n_decode, self.nd_tok
        out = self.out if out is None else out
        if cu_seqlens_host is not None or state_indices_host is not None:
            if cu_seqlens_host is None or state_indices_host is None or (
                    self.N > nd and cu_seqlens_prefill_host is None):
                raise B.GdnError(B.GDN_ERR_INVALID_ARGUMENT, "GDN_ERR_INVALID_ARGUMENT",
                                 "incomplete GDN prefill metadata")
            self.validate(cu_seqlens_host, state_indices_host, cu_seqlens_prefill_host,
                          has_initial_state_host, state_slots=state_pool.shape[0])
        host = cu_seqlens_host is not None
        B.gdn_prepare(mixed_qkv, conv_weight, a_raw, b_raw, A_log, dt_bias, cu_seqlens, conv_pool,
                      self.q, self.k, self.v, self.g, self.beta, Hk=self.Hk, Hv=self.Hv,
                      Dk=self.Dk, Dv=self.Dv, K=self.K, state_indices=state_indices,
                      has_initial_state=has_initial_state, apply_qk_l2norm=self.norm,
                      cu_seqlens_host=cu_seqlens_host if host else None,
                      state_indices_host=state_indices_host if host else None,
                      stream=stream)
        if nd > 0:
            B.gdn_decode(self.q[:ndt], self.k[:ndt], self.v[:ndt], self.g[:ndt],
                         self.beta[:ndt], state_pool, out[:ndt], scale=self.scale,
                         state_indices=state_indices[:nd],
                         state_indices_host=state_indices_host[:nd] if host else None,
                         stream=stream)
        if self.N > nd:
            B.gdn_prefill_varlen(self.q[ndt:], self.k[ndt:], self.v[ndt:], self.g[ndt:],
                                 self.beta[ndt:], state_pool, cu_seqlens_prefill,
                                 out[ndt:], scale=self.scale,
                                 state_indices=state_indices[nd:],
                                 has_initial_state=(None if has_initial_state is None
                                                    else has_initial_state[nd:]),
                                 cu_seqlens_host=cu_seqlens_prefill_host if host else None,
                                 state_indices_host=state_indices_host[nd:] if host else None,
                                 algo=self.algo, workspace=self.workspace, stream=stream)
        return out


class GdnHostPipeline:
    """Steps fed from and drained to pinned host memory, pipelined over three
    streams: step i's inputs are copied in while step i - 1 computes and step
    i - 1's output is copied out while step i computes.  Two device buffers of
    each per-step input and of the output alternate between steps; events keep
    a buffer from being refilled before the compute that reads it (or the copy
    that drains it) is done.

    ``host_inputs`` passed to ``submit`` hold the per-step tensors by name:
    mixed_qkv, a_raw, b_raw, cu_seqlens, state_indices, has_initial_state and
    cu_seqlens_prefill (pinned, the shapes of the first call).  The weights and
    the state and conv pools stay on the device across steps."""

    INPUTS = ("mixed_qkv", "a_raw", "b_raw", "cu_seqlens", "state_indices", "has_initial_state",
              "cu_seqlens_prefill")

    def __init__(self, step: GdnStep, device):
        self.step = step
        self.dev = torch.device(device)
        self.s_in = torch.cuda.Stream(device=self.dev)
        self.s_run = torch.cuda.Stream(device=self.dev)
        self.s_out = torch.cuda.Stream(device=self.dev)
        self.bufs = None
        self.outs = [torch.empty_like(step.out) for _ in range(2)]
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_run = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        self.n = 0

    def submit(self, host_inputs, host_out, conv_weight, A_log, dt_bias, state_pool, conv_pool):
        """Enqueues one step (asynchronous); host_out receives its output."""
        if self.bufs is None:
            self.bufs = [{k: torch.empty(host_inputs[k].shape, dtype=host_inputs[k].dtype,
                                         device=self.dev) for k in self.INPUTS}
                         for _ in range(2)]
        b, i = self.n % 2, self.n
        d = self.bufs[b]
        with torch.cuda.stream(self.s_in):
            if i >= 2:  # step i - 2 has read these buffers
                self.s_in.wait_event(self.ev_run[b])
            for k in self.INPUTS:
                d[k].copy_(host_inputs[k], non_blocking=True)
            self.ev_in[b].record(self.s_in)
        self.s_run.wait_event(self.ev_in[b])
        if i >= 2:  # step i - 2's output has been copied out of this buffer
            self.s_run.wait_event(self.ev_out[b])
        self.step.run(d["mixed_qkv"], d["a_raw"], d["b_raw"], conv_weight, A_log, dt_bias,
                      d["cu_seqlens"], d["state_indices"], d["has_initial_state"], state_pool,
                      conv_pool, d["cu_seqlens_prefill"], stream=self.s_run, out=self.outs[b])
        self.ev_run[b].record(self.s_run)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev_run[b])
            host_out.copy_(self.outs[b], non_blocking=True)
            self.ev_out[b].record(self.s_out)
        self.n += 1

    def synchronize(self):
        for s in (self.s_in, self.s_run, self.s_out):
            s.synchronize()


def mixed_step(mixed_qkv, a_raw, b_raw, conv_weight, A_log, dt_bias, cu_seqlens, state_indices,
               has_initial_state, state_pool, conv_pool, *, n_decode: int, Hk: int, Hv: int,
               Dk: int, Dv: int, K: int, cu_seqlens_prefill=None, scale: float = -1.0,
               algo: int = B.GDN_PREFILL_AUTO, stream=None) -> torch.Tensor:
    """Allocating one-shot form of GdnStep.run; returns out [T, Hv, Dv].  It
    copies the metadata to the host (a synchronisation) and checks the
    mixed-step contract before launching anything."""
    T = mixed_qkv.shape[0]
    N = cu_seqlens.numel() - 1
    step = GdnStep(T, N, n_decode, Hk, Hv, Dk, Dv, K, mixed_qkv.dtype, mixed_qkv.device,
                   scale=scale, algo=algo)
    host = {"cu_seqlens_host": cu_seqlens.cpu(), "state_indices_host": state_indices.cpu(),
            "has_initial_state_host": (None if has_initial_state is None
                                       else has_initial_state.cpu()),
            "cu_seqlens_prefill_host": (None if cu_seqlens_prefill is None
                                        else cu_seqlens_prefill.cpu())}
    return step.run(mixed_qkv, a_raw, b_raw, conv_weight, A_log, dt_bias, cu_seqlens,
                    state_indices, has_initial_state, state_pool, conv_pool,
                    cu_seqlens_prefill=cu_seqlens_prefill, stream=stream, **host).clone()
