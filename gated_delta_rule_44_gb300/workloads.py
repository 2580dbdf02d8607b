"""Seeded synthetic inputs for the GDN layer.

This module only draws random numbers and lays out metadata; it holds none of
the method's arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.  Every tensor is drawn on the CPU with a ``torch.Generator`` seeded by
the workload's seed, in the order the fields are listed in ``make_workload``.

Distributions: ``N(mu, s)`` means mean mu and STANDARD DEVIATION s (the
``torch.normal(mean, std)`` convention); ``U(a, b)`` is uniform on [a, b).

The five named workloads (``WORKLOADS``) are the layer's synthetic benchmark
shapes:
  tiny_f32     T=64 one sequence, Hk=2 Hv=4 Dk=Dv=32 K=4, f32, zero initial state
  decode_b256  256 single-token sequences, Hk=16 Hv=32 D=128 K=4, bf16, 512-slot
               f32 state pool N(0,0.02) gathered by a random permutation
  prefill_4k   one 4096-token sequence, Hk=16 Hv=32 D=128, bf16, zero state
  varlen_8     8 sequences of length U[512, 8192], bf16, N(0,0.02) initial
               states and N(0,1) conv tails carried in
  mixed_hv64   512 decodes then 4 new 2048-token prefills, Hk=16 Hv=64 D=128,
               bf16, 1024-slot pool
The gates are drawn alike everywhere: a,b ~ N(0,1); A_log = log U(1,16);
dt_bias ~ N(0,0.5); conv_weight ~ N(0,1/4); mixed_qkv ~ N(0,1).
A "weak-decay twin" redraws A_log = log U(0.01, 0.1) (g near -0.05 per token)
so that the carried state is not forgotten within a token or two.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    T: int
    N: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    K: int
    act_dtype: torch.dtype          # torch.float32 or torch.bfloat16
    n_decode: int                   # leading single-token sequences (mixed step)
    mixed_qkv: torch.Tensor         # [T, C_conv] act dtype
    conv_weight: torch.Tensor       # [C_conv, K] f32
    a_raw: torch.Tensor             # [T, Hv] act dtype
    b_raw: torch.Tensor             # [T, Hv] act dtype
    A_log: torch.Tensor             # [Hv] f32
    dt_bias: torch.Tensor           # [Hv] f32
    cu_seqlens: torch.Tensor        # [N+1] int32
    state_indices: torch.Tensor     # [N] int32 (pool slot per sequence)
    has_initial_state: torch.Tensor  # [N] uint8
    state_pool: torch.Tensor        # [slots, Hv, Dv, Dk] f32
    conv_pool: torch.Tensor         # [slots, C_conv, K-1] f32

    @property
    def C_conv(self) -> int:
        return 2 * self.Hk * self.Dk + self.Hv * self.Dv

    @property
    def slots(self) -> int:
        return self.state_pool.shape[0]

    @property
    def cu_seqlens_prefill(self) -> torch.Tensor:
        """cu_seqlens of the sequences after the first n_decode, rebased to 0."""
        cu = self.cu_seqlens[self.n_decode:]
        return (cu - cu[0]).to(torch.int32)

    @property
    def seqlens(self) -> List[int]:
        cu = self.cu_seqlens.tolist()
        return [cu[i + 1] - cu[i] for i in range(self.N)]


def _normal(gen, shape, std):
    return torch.empty(shape, dtype=torch.float32).normal_(0.0, std, generator=gen)


def _uniform(gen, shape, lo, hi):
    return torch.empty(shape, dtype=torch.float32).uniform_(lo, hi, generator=gen)


def make_workload(name: str, seed: int, seqlens: List[int], Hk: int, Hv: int, Dk: int, Dv: int,
                  K: int = 4, act_dtype: torch.dtype = torch.bfloat16, slots: Optional[int] = None,
                  init_state: bool = True, init_conv: bool = True, n_decode: int = 0,
                  weak_decay: bool = False, state_std: float = 0.02,
                  permute_slots: bool = True, padded: Optional[List[int]] = None,
                  prefill_new: bool = False) -> Workload:
    """Draws one workload.

    seqlens      token count of each sequence, packed in order (decodes first)
    slots        pool size (default: number of sequences)
    init_state   sequences start from their pool state / conv tail (has_initial_state=1)
    n_decode     the first n_decode sequences are single-token decodes
    prefill_new  sequences after the first n_decode start from zero (has_initial_state=0)
    padded       sequence numbers whose state index is -1 (padding rows)

    Draw order: mixed_qkv, conv_weight, a_raw, b_raw, A_log, dt_bias, state_pool,
    conv_pool, slot permutation.
    """
    gen = torch.Generator(device="cpu").manual_seed(seed)
    N = len(seqlens)
    T = int(sum(seqlens))
    C = 2 * Hk * Dk + Hv * Dv
    slots = N if slots is None else slots
    mixed = _normal(gen, (T, C), 1.0).to(act_dtype)
    conv_w = _normal(gen, (C, K), 0.25)
    a_raw = _normal(gen, (T, Hv), 1.0).to(act_dtype)
    b_raw = _normal(gen, (T, Hv), 1.0).to(act_dtype)
    if weak_decay:
        A_log = _uniform(gen, (Hv,), 0.01, 0.1).log_()
    else:
        A_log = _uniform(gen, (Hv,), 1.0, 16.0).log_()
    dt_bias = _normal(gen, (Hv,), 0.5)
    if init_state:
        state_pool = _normal(gen, (slots, Hv, Dv, Dk), state_std)
        conv_pool = _normal(gen, (slots, C, K - 1), 1.0) if init_conv else torch.zeros(
            (slots, C, K - 1))
    else:
        state_pool = torch.zeros((slots, Hv, Dv, Dk))
        conv_pool = torch.zeros((slots, C, K - 1))
    if permute_slots:
        idx = torch.randperm(slots, generator=gen)[:N].to(torch.int32)
    else:
        idx = torch.arange(N, dtype=torch.int32)
    for p in (padded or []):
        idx[p] = -1
    cu = torch.zeros(N + 1, dtype=torch.int32)
    cu[1:] = torch.tensor(seqlens, dtype=torch.int64).cumsum(0).to(torch.int32)
    has_init = torch.full((N,), 1 if init_state else 0, dtype=torch.uint8)
    if prefill_new:
        has_init[n_decode:] = 0
    return Workload(name=name, seed=seed, T=T, N=N, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K,
                    act_dtype=act_dtype, n_decode=n_decode, mixed_qkv=mixed, conv_weight=conv_w,
                    a_raw=a_raw, b_raw=b_raw, A_log=A_log, dt_bias=dt_bias, cu_seqlens=cu,
                    state_indices=idx, has_initial_state=has_init, state_pool=state_pool,
                    conv_pool=conv_pool)


def varlen_8_lengths(seed: int = 3) -> List[int]:
    """Eight lengths drawn U[512, 8192] (inclusive) from their own seeded generator."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(512, 8193, (8,), generator=gen).tolist()


WORKLOADS = ("tiny_f32", "decode_b256", "prefill_4k", "varlen_8", "mixed_hv64")


def named(name: str, weak_decay: bool = False) -> Workload:
    """One of the five named workloads (seed = its position in WORKLOADS)."""
    if name == "tiny_f32":
        return make_workload(name, 0, [64], 2, 4, 32, 32, act_dtype=torch.float32,
                             init_state=False, permute_slots=False, weak_decay=weak_decay)
    if name == "decode_b256":
        return make_workload(name, 1, [1] * 256, 16, 32, 128, 128, slots=512, n_decode=256,
                             weak_decay=weak_decay)
    if name == "prefill_4k":
        return make_workload(name, 2, [4096], 16, 32, 128, 128, init_state=False,
                             permute_slots=False, weak_decay=weak_decay)
    if name == "varlen_8":
        return make_workload(name, 3, varlen_8_lengths(3), 16, 32, 128, 128,
                             weak_decay=weak_decay)
    if name == "mixed_hv64":
        return make_workload(name, 4, [1] * 512 + [2048] * 4, 16, 64, 128, 128, slots=1024,
                             n_decode=512, prefill_new=True, weak_decay=weak_decay)
    raise KeyError(name)
