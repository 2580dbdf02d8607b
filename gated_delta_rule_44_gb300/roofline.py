"""Algorithmic work per launch of each kernel, for roofline fractions.

Bytes are the minimum HBM traffic the operation implies (each input read once,
each output written once); flops count the useful multiply-adds of the chunked
form (2 flops each), triangular products at their triangular size:

  prepare  per token: x row read (C*es) + q,k,v written (C*es) + a,b read
           (2*Hv*es) + g,beta written (2*Hv*4); per sequence: conv tail read
           (C*(K-1)*4, when it has an initial state) + written (same, when live);
           conv weights once (C*K*4).
  decode   per live row: state read + written (2*Hv*Dv*Dk*4) + q,k (2*Hk*Dk*es)
           + v, out (2*Hv*Dv*es) + g,beta (2*Hv*4); padded rows write out only.
  prefill  flops per chunk of L tokens and value head (chunk 64):
           L^2 (3 Dk + 2 Dv) + 6 L Dk Dv
           (K K^T, Q K^T, T.K, T.V, P.U at triangular size; W S^T, Q S^T and
           the state update at full size), i.e. 139,264 flop per token per head
           at Dk = Dv = 128, L = 64.  Bytes: q,k,v,out,g,beta once + state read
           and written once per live sequence.
es = bytes per activation element (2 for bf16, 4 for f32), C = 2 Hk Dk + Hv Dv.
"""
from __future__ import annotations

from typing import Dict, List

CHUNK = 64


def prepare_bytes(seqlens: List[int], live: List[bool], init: List[bool], Hk, Hv, Dk, Dv, K,
                  es) -> int:
    C = 2 * Hk * Dk + Hv * Dv
    T = sum(seqlens)
    b = T * (2 * C * es + 2 * Hv * es + 2 * Hv * 4) + C * K * 4
    for lv, it in zip(live, init):
        b += (C * (K - 1) * 4 if (lv and it) else 0) + (C * (K - 1) * 4 if lv else 0)
    return b


def decode_bytes(live: List[bool], Hk, Hv, Dk, Dv, es) -> int:
    per_live = 2 * Hv * Dv * Dk * 4 + 2 * Hk * Dk * es + 2 * Hv * Dv * es + 2 * Hv * 4
    return sum(per_live if lv else Hv * Dv * es for lv in live)


def prefill_flops(seqlens: List[int], Hv, Dk, Dv, chunk: int = CHUNK) -> int:
    f = 0
    for L in seqlens:
        full, rem = divmod(L, chunk)
        for l in [chunk] * full + ([rem] if rem else []):
            f += l * l * (3 * Dk + 2 * Dv) + 6 * l * Dk * Dv
    return f * Hv


def prefill_bytes(seqlens: List[int], live: List[bool], init: List[bool], Hk, Hv, Dk, Dv,
                  es) -> int:
    T = sum(seqlens)
    b = T * (2 * Hk * Dk * es + 2 * Hv * Dv * es + 2 * Hv * 4)
    for lv, it in zip(live, init):
        b += (Hv * Dv * Dk * 4 if (lv and it) else 0) + (Hv * Dv * Dk * 4 if lv else 0)
    return b


def step_work(w) -> Dict[str, dict]:
    """Per-kernel algorithmic work of one mixed step of workload `w`."""
    es = 2 if str(w.act_dtype).endswith("bfloat16") else 4
    seqlens = w.seqlens
    live = [int(s) >= 0 for s in w.state_indices.tolist()]
    init = [bool(h) for h in w.has_initial_state.tolist()]
    nd = w.n_decode
    out = {"prepare": {"bytes": prepare_bytes(seqlens, live, init, w.Hk, w.Hv, w.Dk, w.Dv, w.K,
                                              es)}}
    if nd > 0:
        out["decode"] = {"bytes": decode_bytes(live[:nd], w.Hk, w.Hv, w.Dk, w.Dv, es)}
    if w.N > nd:
        sl = seqlens[nd:]
        out["prefill"] = {"flops": prefill_flops(sl, w.Hv, w.Dk, w.Dv),
                          "bytes": prefill_bytes(sl, live[nd:], init[nd:], w.Hk, w.Hv, w.Dk,
                                                 w.Dv, es)}
    return out
