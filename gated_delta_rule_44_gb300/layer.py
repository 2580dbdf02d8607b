"""One GDN layer step over a packed batch: the three library calls in order.

Mixed batches follow [qwen3_5.cpp] (vllm.cpp, src/vllm/model_executor/models/
qwen3_5.cpp) ValidateGdnAttentionMetadata and SubView: the decode rows come
first (one token each), then the prefill sequences.  One ``gdn_prepare`` runs
over every token; ``gdn_decode`` then takes rows [0, n_decode) and
``gdn_prefill_varlen`` the rest, with its cu_seqlens rebased to start at 0
(the caller's ``cu_seqlens_prefill``, like the pages' prefill_query_start_loc).
All buffers are torch tensors on one device; everything is asynchronous on the
given stream.
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

    def run(self, mixed_qkv, a_raw, b_raw, conv_weight, A_log, dt_bias, cu_seqlens, state_indices,
            has_initial_state, state_pool, conv_pool, cu_seqlens_prefill=None,
            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        nd, ndt = self.n_decode, self.nd_tok
        B.gdn_prepare(mixed_qkv, conv_weight, a_raw, b_raw, A_log, dt_bias, cu_seqlens, conv_pool,
                      self.q, self.k, self.v, self.g, self.beta, Hk=self.Hk, Hv=self.Hv,
                      Dk=self.Dk, Dv=self.Dv, K=self.K, state_indices=state_indices,
                      has_initial_state=has_initial_state, apply_qk_l2norm=self.norm,
                      stream=stream)
        if nd > 0:
            B.gdn_decode(self.q[:ndt], self.k[:ndt], self.v[:ndt], self.g[:ndt],
                         self.beta[:ndt], state_pool, self.out[:ndt], scale=self.scale,
                         state_indices=state_indices[:nd], stream=stream)
        if self.N > nd:
            B.gdn_prefill_varlen(self.q[ndt:], self.k[ndt:], self.v[ndt:], self.g[ndt:],
                                 self.beta[ndt:], state_pool, cu_seqlens_prefill,
                                 self.out[ndt:], scale=self.scale,
                                 state_indices=state_indices[nd:],
                                 has_initial_state=(None if has_initial_state is None
                                                    else has_initial_state[nd:]),
                                 algo=self.algo, workspace=self.workspace, stream=stream)
        return self.out


def mixed_step(mixed_qkv, a_raw, b_raw, conv_weight, A_log, dt_bias, cu_seqlens, state_indices,
               has_initial_state, state_pool, conv_pool, *, n_decode: int, Hk: int, Hv: int,
               Dk: int, Dv: int, K: int, cu_seqlens_prefill=None, scale: float = -1.0,
               algo: int = B.GDN_PREFILL_AUTO, stream=None) -> torch.Tensor:
    """Allocating one-shot form of GdnStep.run; returns out [T, Hv, Dv]."""
    T = mixed_qkv.shape[0]
    N = cu_seqlens.numel() - 1
    step = GdnStep(T, N, n_decode, Hk, Hv, Dk, Dv, K, mixed_qkv.dtype, mixed_qkv.device,
                   scale=scale, algo=algo)
    return step.run(mixed_qkv, a_raw, b_raw, conv_weight, A_log, dt_bias, cu_seqlens,
                    state_indices, has_initial_state, state_pool, conv_pool,
                    cu_seqlens_prefill=cu_seqlens_prefill, stream=stream).clone()
