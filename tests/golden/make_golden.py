"""Writes tests/golden/tiny_f32_oracle.txt: summary values of the ORACLE on the
tiny_f32 workload (T=64, Hk=2, Hv=4, Dk=Dv=32, K=4, f32, zero initial state,
seed 0) -- a regression guard, so that any change to the oracle's arithmetic
shows up as a diff of this file.  Calls only oracle/ and the workload
generator.  Run:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gated_delta_rule_44_gb300 import workloads as W  # noqa: E402


def compute():
    w = W.named("tiny_f32")
    conv = w.conv_pool.numpy().copy()
    prep = oracle.prepare_varlen(w.mixed_qkv.numpy(), w.conv_weight.numpy(), conv,
                                 w.a_raw.numpy(), w.b_raw.numpy(), w.A_log.numpy(),
                                 w.dt_bias.numpy(), w.cu_seqlens.numpy(), w.Hk, w.Hv, w.Dk, w.Dv,
                                 w.K, state_indices=w.state_indices.numpy(),
                                 has_initial_state=w.has_initial_state.numpy(), nthreads=1)
    pool = w.state_pool.numpy().copy()
    out = oracle.gdn_varlen(prep["q"], prep["k"], prep["v"], prep["g"], prep["beta"], pool,
                            w.cu_seqlens.numpy(), 1.0 / np.sqrt(w.Dk),
                            state_indices=w.state_indices.numpy(),
                            has_initial_state=w.has_initial_state.numpy(), nthreads=1)
    vals = {}
    for name, arr in (("q", prep["q"]), ("k", prep["k"]), ("v", prep["v"]), ("g", prep["g"]),
                      ("beta", prep["beta"]), ("out", out), ("state", pool), ("conv_tail", conv)):
        a = arr.astype(np.float64)
        vals[f"{name}.sum"] = float(a.sum())
        vals[f"{name}.abssum"] = float(np.abs(a).sum())
        flat = a.reshape(-1)
        for i in (0, flat.size // 3, flat.size - 1):
            vals[f"{name}[{i}]"] = float(flat[i])
    return vals


if __name__ == "__main__":
    vals = compute()
    with open(os.path.join(HERE, "tiny_f32_oracle.txt"), "w") as fh:
        fh.write("# Oracle (f32) on the tiny_f32 workload; written by tests/golden/make_golden.py\n")
        fh.write("# (oracle/ only).  Regression guard for the oracle's own arithmetic.\n")
        for k, v in vals.items():
            fh.write(f"{k} {v!r}\n")
