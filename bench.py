#!/usr/bin/env python3
"""Benchmark of the GDN layer step on GB300.

A step is one pass of the whole hot path over one batch: gdn_prepare over every
token (conv1d + SiLU + split + q/k L2 norm + gates, conv tails in the pool),
gdn_decode on the leading single-token rows and gdn_prefill_varlen (chunked
tensor-core form) on the prefill sequences.  The default workload is the mixed
serving step (512 decodes + 4 new 2048-token prefills, Hk=16 Hv=64 Dk=Dv=128,
bf16 activations, f32 state pool of 1024 slots): the one configuration that
runs every step of the path.  Inputs are seeded synthetic data already resident
in HBM; the working set (state rows streamed by the decodes, 214 MB of
mixed_qkv) is far larger than the 129 MB L2, so no flush is inserted.

Prints ONE JSON line (rank 0).  Multi-GPU: one process per GPU under torchrun;
each rank runs its own replica of the workload (the layer shards by sequence
and head with no exchange), so scaling is weak and the value counts the tokens
of all ranks over the slowest rank's time.

--impl reference times the CPU oracle (the plain C++ restatement of the
pages' CPU code) over whole steps of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN tokens/sec (decode, prefill) and % of HBM / bf16 tensor roofline"
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed_hv64")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the single-kernel decode / prefill workloads")
    ap.add_argument("--algo", type=int, default=0, help="prefill algorithm (0 auto)")
    ap.add_argument("--extra-only", default=None,
                    choices=["kda_prefill_4k", "kda_decode_b256", "spec_decode_r128x4",
                             "spec_prepare_r128x4", "packed_decode_b256"],
                    help="time one of the extra measurements alone (a small case for profiling)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---- clocks ------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.fh = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.flush()
        self.fh.seek(0)
        rows = [r.split(",") for r in self.fh.read().strip().splitlines() if r.strip()]
        os.unlink(self.fh.name)
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 10]
        if self.bus_id:
            mine = [r for r in rows if r[1].lower().endswith(self.bus_id[-12:])]
            rows = mine or rows
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v == "Active"})
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---- our arm ---------------------------------------------------------------------

def dev_inputs(w, dev):
    return dict(mixed_qkv=w.mixed_qkv.to(dev), conv_weight=w.conv_weight.to(dev),
                a_raw=w.a_raw.to(dev), b_raw=w.b_raw.to(dev), A_log=w.A_log.to(dev),
                dt_bias=w.dt_bias.to(dev), cu_seqlens=w.cu_seqlens.to(dev),
                state_indices=w.state_indices.to(dev),
                has_initial_state=w.has_initial_state.to(dev),
                state_pool=w.state_pool.to(dev), conv_pool=w.conv_pool.to(dev),
                cu_seqlens_prefill=w.cu_seqlens_prefill.to(dev))


def run_step_events(step, d, stream, evs):
    """One step with an event between every library call (on the launch stream)."""
    import gated_delta_rule_44_gb300.binding as B
    nd, ndt = step.n_decode, step.nd_tok
    evs[0].record(stream)
    B.gdn_prepare(d["mixed_qkv"], d["conv_weight"], d["a_raw"], d["b_raw"], d["A_log"],
                  d["dt_bias"], d["cu_seqlens"], d["conv_pool"], step.q, step.k, step.v, step.g,
                  step.beta, Hk=step.Hk, Hv=step.Hv, Dk=step.Dk, Dv=step.Dv, K=step.K,
                  state_indices=d["state_indices"], has_initial_state=d["has_initial_state"],
                  stream=stream)
    evs[1].record(stream)
    if nd > 0:
        B.gdn_decode(step.q[:ndt], step.k[:ndt], step.v[:ndt], step.g[:ndt], step.beta[:ndt],
                     d["state_pool"], step.out[:ndt], state_indices=d["state_indices"][:nd],
                     stream=stream)
    evs[2].record(stream)
    if step.N > nd:
        B.gdn_prefill_varlen(step.q[ndt:], step.k[ndt:], step.v[ndt:], step.g[ndt:],
                             step.beta[ndt:], d["state_pool"], d["cu_seqlens_prefill"],
                             step.out[ndt:], state_indices=d["state_indices"][nd:],
                             has_initial_state=d["has_initial_state"][nd:], algo=step.algo,
                             workspace=step.workspace, stream=stream)
    evs[3].record(stream)


def time_workload(w, dev, steps, warmup, algo, dist=None, clocks=None):
    """Device-timed K steps; returns timing dict incl. per-kernel averages."""
    import torch
    import gated_delta_rule_44_gb300.binding as B
    from gated_delta_rule_44_gb300.layer import GdnStep
    d = dev_inputs(w, dev)
    step = GdnStep(w.T, w.N, w.n_decode, w.Hk, w.Hv, w.Dk, w.Dv, w.K, w.act_dtype, dev,
                   algo=algo)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                  for _ in range(steps + warmup)]
        for i in range(warmup):
            run_step_events(step, d, stream, evsets[i])
        stream.synchronize()
        B.gdn_read_device_status(stream)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        if clocks is not None:
            clocks.start()
            time.sleep(0.3)
        launches0 = B.gdn_launch_count()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(warmup, warmup + steps):
            run_step_events(step, d, stream, evsets[i])
        t1.record(stream)
        launches = B.gdn_launch_count() - launches0
        stream.synchronize()
        torch.cuda.synchronize(dev)
        clk = clocks.stop() if clocks is not None else None
        if dist is not None:
            dist.barrier()
        B.gdn_read_device_status(stream)
    total_ms = t0.elapsed_time(t1)
    per = {"prepare": [], "decode": [], "prefill": []}
    for i in range(warmup, warmup + steps):
        e = evsets[i]
        per["prepare"].append(e[0].elapsed_time(e[1]))
        per["decode"].append(e[1].elapsed_time(e[2]))
        per["prefill"].append(e[2].elapsed_time(e[3]))
    avg = {k: sum(v) / len(v) for k, v in per.items()}
    del d, step
    torch.cuda.empty_cache()
    return dict(total_ms=total_ms, ms_per_step=total_ms / steps, kernel_ms=avg,
                launches=launches, clocks=clk)


def kernel_report(w, kernel_ms, peaks):
    from gated_delta_rule_44_gb300 import roofline as R
    work = R.step_work(w)
    rep = {}
    for name, wk in work.items():
        ms = kernel_ms.get(name, 0.0)
        if ms <= 0:
            continue
        entry = {"avg_us": round(ms * 1e3, 2)}
        gbs = wk["bytes"] / (ms * 1e-3) / 1e9
        entry["algorithmic_bytes"] = wk["bytes"]
        entry["achieved_gbs"] = round(gbs, 1)
        entry["hbm_frac_of_measured"] = round(gbs / peaks["hbm"], 4)
        entry["hbm_frac_of_8tbs"] = round(gbs / 8000.0, 4)
        if "flops" in wk:
            tf = wk["flops"] / (ms * 1e-3) / 1e12
            entry["algorithmic_flops"] = wk["flops"]
            entry["achieved_tflops"] = round(tf, 2)
            entry["tensor_frac_of_measured"] = round(tf / peaks["bf16"], 4)
        rep[name] = entry
    return rep, work


# DRAM bytes (read + write) per library call, measured with ncu on a GB300
# (dram__bytes_read.sum + dram__bytes_write.sum summed over the call's launches),
# keyed by (call, workload), with the sha256 of the kernel sources they were
# measured on (concatenated in the order listed): once a source changes the
# figure no longer applies and the line reports null.  mixed_hv64 is too large
# to capture under ncu's replay, so its figures are scaled from smaller cases
# of the same kernels: the decode by the row-heads processed (x4; every byte
# of that launch is per row-head), the fused prefill by the call's algorithmic
# bytes (varlen_8's traffic was 0.981 of its algorithmic bytes; the per-token
# share of key and value heads differs between the two workloads, so token-heads
# would not scale it).
_DECODE_SRC = (("gdn_recurrent.cu", "gdn_rowstep.cuh", "gdn_math.cuh"),
               "27a316189865ac53a673efa7b8dd7d8cac0c7b20a4885acb1593f84a0d92486b")
_FUSED_SRC = (("gdn_fused.cu", "gdn_chunk_common.cuh", "tcgen05.cuh"),
              "58e72a3ea6a4cc1ff4d8b4f047b10bcbf6fff1c2f1e9a49892082aeb670e871e")
_CHUNKED_SRC = (("gdn_chunked.cu", "gdn_chunk_common.cuh", "tcgen05.cuh"),
                "d52e0bff59df7a9a5c1e8b0a9d0701657d3c9cdd0d30d4ee728c9482d8f1080a")
MEASURED_TRAFFIC = {
    ("prefill", "prefill_4k"): (244.0e6,) + _CHUNKED_SRC +
                               ("the call's 4 chunk_prep + 4 chunk_scan launches; ncu flushes L2 "
                                "between them, so blob writes still in L2 are not counted",),
    ("prefill", "varlen_8"): (633.9e6,) + _FUSED_SRC +
                             ("the fused_prefill launch (the schedule kernel's few KB not counted)",),
    ("prefill", "mixed_hv64"): (349.7e6,) + _FUSED_SRC +
                               ("varlen_8's fused launch scaled by algorithmic bytes (x0.552)",),
    ("decode", "decode_b256"): (1017.8e6,) + _DECODE_SRC + ("one decode launch",),
    ("decode", "mixed_hv64"): (4071.2e6,) + _DECODE_SRC + ("decode_b256's launch x 4 (row-heads)",),
}


def measured_traffic(call, workload):
    """(bytes, how) for the call on the workload when the kernel source still
    matches the one measured, else (None, reason)."""
    import hashlib
    ent = MEASURED_TRAFFIC.get((call, workload))
    if ent is None:
        return None, "not captured"
    nbytes, srcs, sha, how = ent
    h = hashlib.sha256()
    for src in srcs:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                            "gated_delta_rule_44_gb300", "csrc", src)
        with open(path, "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != sha:
        return None, f"{' + '.join(srcs)} changed since the capture"
    return int(nbytes), how


def roofline_entry(w, kernel_ms, peaks):
    rep, work = kernel_report(w, kernel_ms, peaks)
    dom = max(rep, key=lambda k: rep[k]["avg_us"])
    r = rep[dom]
    traffic, how = measured_traffic(dom, w.name)
    if "flops" in work[dom]:
        ach = r["achieved_tflops"]
        return dom, {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peaks["bf16"],
                     "unit": "TFLOP/s", "frac": round(ach / peaks["bf16"], 4),
                     "traffic": traffic, "traffic_source": how,
                     "peak_source": peaks["source"] + " (burst)"}, rep
    ach = r["achieved_gbs"]
    return dom, {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm"],
                 "unit": "GB/s", "frac": round(ach / peaks["hbm"], 4), "traffic": traffic,
                 "traffic_source": how, "peak_source": peaks["source"]}, rep


def time_gated_rmsnorm(w, dev, peaks, iters=20):
    """gdn_gated_rmsnorm on the step's output shape [T, Hv, Dv] (bf16; the
    step after the recurrence, not part of the GDN step timed above).
    Algorithmic bytes: core and z read, out written once (2 bytes each)."""
    import torch
    from gated_delta_rule_44_gb300 import binding as B
    g = torch.Generator().manual_seed(17)
    shape = (w.T, w.Hv, w.Dv)
    core = torch.randn(shape, generator=g).to(torch.bfloat16).to(dev)
    z = torch.randn(shape, generator=g).to(torch.bfloat16).to(dev)
    wt = (torch.rand(w.Dv, generator=g) + 0.5).to(torch.bfloat16).to(dev)
    out = torch.empty_like(core)
    s = torch.cuda.current_stream(dev)
    for _ in range(3):
        B.gdn_gated_rmsnorm(core, z, wt, out, stream=s)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(s)
    for _ in range(iters):
        B.gdn_gated_rmsnorm(core, z, wt, out, stream=s)
    e1.record(s)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) / iters * 1e3
    nbytes = core.numel() * 2 * 3 + w.Dv * 2
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"shape": list(shape), "avg_us": round(us, 2), "algorithmic_bytes": nbytes,
            "achieved_gbs": round(gbs, 1), "hbm_frac_of_measured": round(gbs / peaks["hbm"], 4)}


def time_out_norm_routes(w, dev, algo, iters=10):
    """The step's recurrence calls (decode rows, then the prefill) followed by
    the gated RMSNorm of their output, three ways: the norm as its own call
    after them; the out_norm option of the calls (the norm kernel after each);
    and the option with the decode's norm inside the decode kernel.
    Gate rows z [T, Hv*Dv] and weight [Dv] bf16, seeded; q, k, v, g, beta are
    the step's own prepare outputs.  Reports each route's average time."""
    import torch
    from gated_delta_rule_44_gb300 import binding as B
    from gated_delta_rule_44_gb300.layer import GdnStep
    d = dev_inputs(w, dev)
    step = GdnStep(w.T, w.N, w.n_decode, w.Hk, w.Hv, w.Dk, w.Dv, w.K, w.act_dtype, dev, algo=algo)
    s = torch.cuda.current_stream(dev)
    B.gdn_prepare(d["mixed_qkv"], d["conv_weight"], d["a_raw"], d["b_raw"], d["A_log"],
                  d["dt_bias"], d["cu_seqlens"], d["conv_pool"], step.q, step.k, step.v, step.g,
                  step.beta, Hk=step.Hk, Hv=step.Hv, Dk=step.Dk, Dv=step.Dv, K=step.K,
                  state_indices=d["state_indices"], has_initial_state=d["has_initial_state"],
                  stream=s)
    g = torch.Generator().manual_seed(23)
    z = torch.randn(w.T, w.Hv * w.Dv, generator=g).to(torch.bfloat16).to(dev)
    wt = (torch.rand(w.Dv, generator=g) + 0.5).to(torch.bfloat16).to(dev)
    normed = torch.empty_like(step.out)
    nd, ndt = step.n_decode, step.nd_tok

    def calls(route):
        fused = route != "separate_us"
        kw = {}
        if nd > 0:
            if fused:
                kw = dict(norm_z=z[:ndt], norm_weight=wt,
                          norm_in_kernel=route == "decode_in_kernel_us")
            B.gdn_decode(step.q[:ndt], step.k[:ndt], step.v[:ndt], step.g[:ndt],
                         step.beta[:ndt], d["state_pool"], step.out[:ndt],
                         state_indices=d["state_indices"][:nd], stream=s, **kw)
        if step.N > nd:
            if fused:
                kw = dict(norm_z=z[ndt:], norm_weight=wt)
            B.gdn_prefill_varlen(step.q[ndt:], step.k[ndt:], step.v[ndt:], step.g[ndt:],
                                 step.beta[ndt:], d["state_pool"], d["cu_seqlens_prefill"],
                                 step.out[ndt:], state_indices=d["state_indices"][nd:],
                                 has_initial_state=d["has_initial_state"][nd:], algo=step.algo,
                                 workspace=step.workspace, stream=s, **kw)
        if not fused:
            B.gdn_gated_rmsnorm(step.out, z, wt, normed, stream=s)

    res = {}
    for route in ("separate_us", "out_norm_option_us", "decode_in_kernel_us"):
        for _ in range(3):
            calls(route)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(s)
        for _ in range(iters):
            calls(route)
        e1.record(s)
        torch.cuda.synchronize(dev)
        res[route] = round(e0.elapsed_time(e1) / iters * 1e3, 2)
    B.gdn_read_device_status(s)
    del d, step
    torch.cuda.empty_cache()
    return {"calls": "decode + prefill + gated RMSNorm of the output", **res}


def time_kda_decode(dev, peaks, B_=256, Hk=16, Hv=32, D=128, slots=512, iters=10):
    """gdn_kda_varlen on decode_b256's shape (256 one-token sequences, a
    512-slot f32 pool, bf16 activations).  Algorithmic bytes: every live state
    row read and written once, plus q, k, v, out (bf16), g (f32 per key
    channel) and beta."""
    import torch
    from gated_delta_rule_44_gb300 import binding as B
    gen = torch.Generator().manual_seed(23)
    q = (torch.randn(B_, Hk, D, generator=gen) / D ** 0.5).to(torch.bfloat16).to(dev)
    k = (torch.randn(B_, Hk, D, generator=gen) / D ** 0.5).to(torch.bfloat16).to(dev)
    v = torch.randn(B_, Hv, D, generator=gen).to(torch.bfloat16).to(dev)
    g = (-torch.rand(B_, Hv, D, generator=gen) * 0.3).to(dev)
    beta = (torch.rand(B_, Hv, generator=gen) * 0.8 + 0.1).to(dev)
    pool = (torch.randn(slots, Hv, D, D, generator=gen) * 0.02).to(dev)
    sidx = torch.randperm(slots, generator=gen)[:B_].to(torch.int32).to(dev)
    cu = torch.arange(B_ + 1, dtype=torch.int32).to(dev)
    out = torch.empty(B_, Hv, D, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream(dev)

    def call():
        B.gdn_kda_varlen(q, k, v, g, beta, pool, cu, out, state_indices=sidx, stream=s)

    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(s)
    for _ in range(iters):
        call()
    e1.record(s)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) / iters * 1e3
    nbytes = (B_ * Hv * D * D * 4 * 2 + 2 * B_ * Hk * D * 2 + 2 * B_ * Hv * D * 2
              + B_ * Hv * D * 4 + B_ * Hv * 4)
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"tokens_per_s": round(B_ / (us * 1e-6), 1), "avg_us": round(us, 2),
            "algorithmic_bytes": nbytes, "achieved_gbs": round(gbs, 1),
            "hbm_frac_of_measured": round(gbs / peaks["hbm"], 4)}


def time_kda_prefill(dev, peaks, T=4096, Hk=16, Hv=32, D=128, iters=5):
    """gdn_kda_varlen on the single-sequence prefill shape (one 4096-token
    sequence, 16 / 32 heads of 128, bf16, g = -U(0, 0.3) per key channel),
    both forms: the chunked tensor-core one (its two launches) and the
    recurrent one.  Algorithmic FLOPs: the chunk-64 form's contractions, as
    for the scalar-decay prefill."""
    import torch
    from gated_delta_rule_44_gb300 import binding as B
    from gated_delta_rule_44_gb300 import roofline as R
    gen = torch.Generator().manual_seed(29)
    q = (torch.randn(T, Hk, D, generator=gen) / D ** 0.5).to(torch.bfloat16).to(dev)
    k = (torch.randn(T, Hk, D, generator=gen) / D ** 0.5).to(torch.bfloat16).to(dev)
    v = torch.randn(T, Hv, D, generator=gen).to(torch.bfloat16).to(dev)
    g = (-torch.rand(T, Hv, D, generator=gen) * 0.3).to(dev)
    beta = (torch.rand(T, Hv, generator=gen) * 0.8 + 0.1).to(dev)
    pool = (torch.randn(1, Hv, D, D, generator=gen) * 0.02).to(dev)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    out = torch.empty(T, Hv, D, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(B.gdn_kda_workspace_bytes(T, 1, Hv, D, D, 1, B.GDN_PREFILL_CHUNKED),
                     dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev)
    res = {"shape": [T, Hk, Hv, D]}
    for name, algo in (("chunked", B.GDN_PREFILL_CHUNKED), ("recurrent", B.GDN_PREFILL_RECURRENT)):
        def call():
            B.gdn_kda_varlen(q, k, v, g, beta, pool, cu, out, algo=algo,
                             workspace=ws if algo == B.GDN_PREFILL_CHUNKED else None, stream=s)
        for _ in range(3):
            call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(s)
        for _ in range(iters):
            call()
        e1.record(s)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) / iters * 1e3
        res[name] = {"avg_us": round(us, 2), "tokens_per_s": round(T / (us * 1e-6), 1)}
    B.gdn_read_device_status(s)
    flops = R.prefill_flops([T], Hv, D, D)
    tf = flops / (res["chunked"]["avg_us"] * 1e-6) / 1e12
    res["chunked"].update({"algorithmic_flops": flops, "achieved_tflops": round(tf, 2),
                           "tensor_frac_of_measured": round(tf / peaks["bf16"], 4)})
    return res


def time_spec_decode(dev, peaks, n_reqs=128, num_cols=4, Hk=16, Hv=32, D=128, slots=1024,
                     iters=10):
    """gdn_spec_decode on a multi-token-prediction decode: 128 requests x 4
    draft tokens (num_cols 4), a 1024-slot f32 pool, bf16 activations, each
    request resuming from a random accepted column.  Algorithmic bytes: per
    (request, head) one state read and one state write per draft token, plus
    q, k, v, out (bf16), g, beta (f32) and the metadata."""
    import torch
    from gated_delta_rule_44_gb300 import binding as B
    gen = torch.Generator().manual_seed(29)
    T = n_reqs * num_cols
    q = (torch.randn(T, Hk, D, generator=gen) / D ** 0.5).to(torch.bfloat16).to(dev)
    k = (torch.randn(T, Hk, D, generator=gen) / D ** 0.5).to(torch.bfloat16).to(dev)
    v = torch.randn(T, Hv, D, generator=gen).to(torch.bfloat16).to(dev)
    g = (-torch.rand(T, Hv, generator=gen) * 0.3).to(dev)
    beta = (torch.rand(T, Hv, generator=gen) * 0.8 + 0.1).to(dev)
    pool = (torch.randn(slots, Hv, D, D, generator=gen) * 0.02).to(dev)
    sidx = torch.randperm(slots, generator=gen)[:T].reshape(n_reqs, num_cols)
    sidx = sidx.to(torch.int32).to(dev)
    nat = torch.randint(1, num_cols + 1, (n_reqs,), generator=gen, dtype=torch.int32).to(dev)
    cu = (torch.arange(n_reqs + 1, dtype=torch.int32) * num_cols).to(dev)
    out = torch.empty(T, Hv, D, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream(dev)

    def call():
        B.gdn_spec_decode(q, k, v, g, beta, pool, cu, sidx, nat, out, stream=s)

    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(s)
    for _ in range(iters):
        call()
    e1.record(s)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) / iters * 1e3
    state = Hv * D * D * 4
    nbytes = (n_reqs * state * (1 + num_cols) + 2 * T * Hk * D * 2 + 2 * T * Hv * D * 2
              + 2 * T * Hv * 4 + 4 * (n_reqs * (num_cols + 2) + 1))
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"tokens_per_s": round(T / (us * 1e-6), 1), "avg_us": round(us, 2),
            "requests": n_reqs, "num_cols": num_cols, "algorithmic_bytes": nbytes,
            "achieved_gbs": round(gbs, 1), "hbm_frac_of_measured": round(gbs / peaks["hbm"], 4)}


def time_spec_prepare(dev, peaks, n_reqs=128, max_q=4, Hk=16, Hv=32, D=128, K=4, slots=1024,
                      iters=10):
    """gdn_spec_prepare on the same multi-token-prediction step (128 requests
    x 4 drafts, conv rows of (K-1) + (max_q-1) = 6 raw inputs per channel).
    Algorithmic bytes: mixed_qkv read and q, k, v written once (bf16), each
    request's conv row read and written once (f32), the gate inputs (bf16)
    and outputs (f32), the conv weights."""
    import torch
    from gated_delta_rule_44_gb300 import binding as B
    gen = torch.Generator().manual_seed(31)
    T, C, width = n_reqs * max_q, 2 * Hk * D + Hv * D, (K - 1) + (max_q - 1)
    x = torch.randn(T, C, generator=gen).to(torch.bfloat16).to(dev)
    wconv = (torch.randn(C, K, generator=gen) * 0.4).to(dev)
    a = torch.randn(T, Hv, generator=gen).to(torch.bfloat16).to(dev)
    b = torch.randn(T, Hv, generator=gen).to(torch.bfloat16).to(dev)
    A_log, dt_bias = torch.zeros(Hv, device=dev), torch.zeros(Hv, device=dev)
    pool = torch.randn(slots, C, width, generator=gen).to(dev)
    idx = torch.randperm(slots, generator=gen)[:n_reqs].to(torch.int32).to(dev)
    nat = torch.randint(1, max_q + 1, (n_reqs,), generator=gen, dtype=torch.int32).to(dev)
    cu = (torch.arange(n_reqs + 1, dtype=torch.int32) * max_q).to(dev)
    q = torch.empty(T, Hk, D, dtype=torch.bfloat16, device=dev)
    k = torch.empty_like(q)
    v = torch.empty(T, Hv, D, dtype=torch.bfloat16, device=dev)
    g = torch.empty(T, Hv, device=dev)
    beta = torch.empty_like(g)
    s = torch.cuda.current_stream(dev)

    def call():
        B.gdn_spec_prepare(x, wconv, a, b, A_log, dt_bias, cu, pool, idx, nat, q, k, v, g, beta,
                           Hk=Hk, Hv=Hv, Dk=D, Dv=D, K=K, stream=s)

    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(s)
    for _ in range(iters):
        call()
    e1.record(s)
    torch.cuda.synchronize(dev)
    host_us = e0.elapsed_time(e1) / iters * 1e3
    # The kernel is shorter than one call's host-side marshalling, so the loop
    # above measures the host.  Device time: the same calls captured in a
    # CUDA graph and replayed.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cs = torch.cuda.current_stream(dev)
        for _ in range(iters):
            B.gdn_spec_prepare(x, wconv, a, b, A_log, dt_bias, cu, pool, idx, nat, q, k, v, g,
                               beta, Hk=Hk, Hv=Hv, Dk=D, Dv=D, K=K, stream=cs)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0.record(s)
    graph.replay()
    e1.record(s)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) / iters * 1e3
    nbytes = (2 * T * C * 2 + 2 * n_reqs * C * width * 4 + 2 * T * Hv * 2 + 2 * T * Hv * 4
              + C * K * 4 + 4 * (2 * n_reqs + 1))
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"tokens_per_s": round(T / (us * 1e-6), 1), "avg_us": round(us, 2),
            "timing": "CUDA graph of the calls", "host_loop_us": round(host_us, 2),
            "requests": n_reqs, "max_q": max_q, "algorithmic_bytes": nbytes,
            "achieved_gbs": round(gbs, 1), "hbm_frac_of_measured": round(gbs / peaks["hbm"], 4)}


def time_packed_decode(dev, peaks, B_=256, Hk=16, Hv=32, D=128, K=4, slots=512, iters=10):
    """gdn_packed_decode on decode_b256's shape: conv update, norm, gates and
    the recurrence in one launch from a packed qkvz row and a b-then-a gate
    row.  Algorithmic bytes: every live state row read and written once, the
    conv tails read and written once, the raw rows (q, k, v channels), the
    gate inputs, out (bf16) and the conv weights."""
    import torch
    from gated_delta_rule_44_gb300 import binding as B
    gen = torch.Generator().manual_seed(37)
    C = 2 * Hk * D + Hv * D
    qkvz = torch.randn(B_, C + Hv * D, generator=gen).to(torch.bfloat16).to(dev)
    wconv = (torch.randn(C, K, generator=gen) * 0.4).to(dev)
    ba = torch.randn(B_, 2 * Hv, generator=gen).to(torch.bfloat16).to(dev)
    a_raw, b_raw = B.packed_ba_views(ba, Hv)
    A_log, dt_bias = torch.zeros(Hv, device=dev), torch.zeros(Hv, device=dev)
    conv = torch.randn(slots, C, K - 1, generator=gen).to(dev)
    pool = (torch.randn(slots, Hv, D, D, generator=gen) * 0.02).to(dev)
    sidx = torch.randperm(slots, generator=gen)[:B_].to(torch.int32).to(dev)
    out = torch.empty(B_, Hv, D, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream(dev)

    def call():
        B.gdn_packed_decode(qkvz, wconv, a_raw, b_raw, A_log, dt_bias, sidx, conv, pool, out,
                            Hk=Hk, Hv=Hv, Dk=D, Dv=D, K=K, stream=s)

    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(s)
    for _ in range(iters):
        call()
    e1.record(s)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) / iters * 1e3
    nbytes = (B_ * Hv * D * D * 4 * 2 + B_ * C * 2 + 2 * B_ * C * (K - 1) * 4
              + B_ * 2 * Hv * 2 + B_ * Hv * D * 2 + C * K * 4 + B_ * 4)
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"tokens_per_s": round(B_ / (us * 1e-6), 1), "avg_us": round(us, 2),
            "algorithmic_bytes": nbytes, "achieved_gbs": round(gbs, 1),
            "hbm_frac_of_measured": round(gbs / peaks["hbm"], 4)}


def time_e2e(w, dev, steps, warmup, algo):
    """Same step through the public API with the step's inputs in pinned host
    memory: every step copies its inputs host -> device and its output
    device -> host inside the timed region (GdnHostPipeline overlaps those
    copies with the neighbouring steps' compute).  The first step's input copy
    and the last step's output copy have nothing to overlap with and are
    included; over K steps they add (H2D + D2H time) / K per step."""
    import torch
    from gated_delta_rule_44_gb300.layer import GdnHostPipeline, GdnStep
    d = dev_inputs(w, dev)
    host_in = {k: getattr(w, k).pin_memory() for k in GdnHostPipeline.INPUTS}
    step = GdnStep(w.T, w.N, w.n_decode, w.Hk, w.Hv, w.Dk, w.Dv, w.K, w.act_dtype, dev,
                   algo=algo)
    out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = out_host.numel() * out_host.element_size()
    pipe = GdnHostPipeline(step, dev)

    def one():
        pipe.submit(host_in, out_host, d["conv_weight"], d["A_log"], d["dt_bias"],
                    d["state_pool"], d["conv_pool"])

    for _ in range(warmup):
        one()
    pipe.synchronize()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(pipe.s_in)
    for _ in range(steps):
        one()
    t1.record(pipe.s_out)  # after the last step's output copy
    pipe.synchronize()
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / steps
    del d, step, pipe
    torch.cuda.empty_cache()
    return {"value": round(w.T / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": "inputs in, outputs out and compute on three streams"}


# ---- CPU oracle baseline -----------------------------------------------------------

def oracle_step(w, nthreads, state_pool, conv_pool):
    """One whole step of the workload on the oracle, timed: the prepare over
    every token, then the recurrence over every sequence (decode rows are
    one-token sequences) and every value head, each parallel over its items on
    `nthreads` host threads.  The pools are updated in place, as the GPU step
    does.  Returns seconds."""
    import numpy as np
    import oracle
    f32 = lambda t: t.float().numpy()
    t0 = time.perf_counter()
    prep = oracle.prepare_varlen(f32(w.mixed_qkv), w.conv_weight.numpy(), conv_pool, f32(w.a_raw),
                                 f32(w.b_raw), w.A_log.numpy(), w.dt_bias.numpy(),
                                 w.cu_seqlens.numpy(), w.Hk, w.Hv, w.Dk, w.Dv, w.K,
                                 state_indices=w.state_indices.numpy(),
                                 has_initial_state=w.has_initial_state.numpy(),
                                 dtype=np.float32, nthreads=nthreads)
    oracle.gdn_varlen(prep["q"], prep["k"], prep["v"], prep["g"], prep["beta"], state_pool,
                      w.cu_seqlens.numpy(), 1.0 / np.sqrt(w.Dk),
                      state_indices=w.state_indices.numpy(),
                      has_initial_state=w.has_initial_state.numpy(), dtype=np.float32,
                      nthreads=nthreads)
    return time.perf_counter() - t0


def oracle_pools(w):
    """Private f32 copies of the workload's state and conv pools."""
    import numpy as np
    return (np.ascontiguousarray(w.state_pool.numpy(), dtype=np.float32).copy(),
            np.ascontiguousarray(w.conv_pool.numpy(), dtype=np.float32).copy())


def oracle_sample_text(w, nthreads, steps):
    return (f"{steps} whole step(s) of the workload on the oracle (C++ f32, {nthreads} host "
            f"threads, parallel over (sequence, value head)): prepare over all {w.T} tokens and "
            f"the recurrence over all {w.N} sequences x {w.Hv} value heads; no extrapolation")


def cpu_baseline(w, nthreads):
    """The oracle as it stands, timed over one whole step of the workload."""
    sp, cp = oracle_pools(w)
    secs = oracle_step(w, nthreads, sp, cp)
    return {"value": round(w.T / secs, 2), "unit": "tokens/s", "cores": nthreads,
            "kind": "oracle", "sample": oracle_sample_text(w, nthreads, 1),
            "seconds": round(secs, 2)}


def workload_config(w, ws):
    """The `config` object of the JSON line; both arms print this same dict."""
    return {"workload": w.name, "tokens_per_step": w.T, "decodes": w.n_decode,
            "prefill_seqlens": w.seqlens[w.n_decode:], "Hk": w.Hk, "Hv": w.Hv, "Dk": w.Dk,
            "Dv": w.Dv, "conv_kernel": w.K, "state_slots": w.slots, "state_dtype": "f32",
            "parallelism": f"replicas{ws}", "l2": "inputs larger than L2 (no flush)"}


def rank_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def slowest_rank_ms(ms, dist, device):
    """The step time of the slowest rank, on every rank (ms itself at N = 1).
    Each rank runs its own replica of the workload, so the whole job's step
    takes as long as its slowest replica."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_rank, ws, ms):
    """Tokens per second of all ranks together (weak scaling: every rank
    processes tokens_per_rank tokens per step)."""
    return tokens_per_rank * ws / (ms * 1e-3)


def main_reference(args):
    """The oracle timed over W untimed then K timed whole steps of the same
    workload on the host cores (rank 0 only)."""
    ws, rank, _ = rank_info()
    if rank != 0:
        return 0
    from gated_delta_rule_44_gb300 import workloads as W
    import oracle
    oracle.build()
    w = W.named(args.workload)
    nthreads = os.cpu_count() or 1
    sp, cp = oracle_pools(w)
    for _ in range(args.warmup):
        oracle_step(w, nthreads, sp, cp)
    secs = [oracle_step(w, nthreads, sp, cp) for _ in range(args.steps)]
    total = sum(secs)
    v = w.T * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(w, ws),
            "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s", "cores": nthreads,
                             "kind": "oracle",
                             "sample": oracle_sample_text(w, nthreads, args.steps)},
            "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return main_reference(args)
    import torch
    ws, rank, local = rank_info()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    import gated_delta_rule_44_gb300.binding as B
    from gated_delta_rule_44_gb300 import workloads as W
    B.lib()
    peaks = load_peaks()
    if args.extra_only is not None:
        fn = {"kda_prefill_4k": time_kda_prefill, "kda_decode_b256": time_kda_decode,
              "spec_decode_r128x4": time_spec_decode, "spec_prepare_r128x4": time_spec_prepare,
              "packed_decode_b256": time_packed_decode}[args.extra_only]
        print(json.dumps({"extra": args.extra_only, "result": fn(dev, peaks)}), flush=True)
        return 0
    w = W.named(args.workload)
    props = torch.cuda.get_device_properties(dev)
    bus = getattr(props, "pci_bus_id", None)
    clocks = ClockSampler(bus) if rank == 0 else None
    res = time_workload(w, dev, args.steps, max(args.warmup, 3), args.algo, dist, clocks)
    ms = slowest_rank_ms(res["ms_per_step"], dist, dev)
    value = whole_job_value(w.T, ws, ms)
    dom, roof, kernels = roofline_entry(w, res["kernel_ms"], peaks)
    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": workload_config(w, ws),
            "prefill_algo": B.gdn_prefill_resolve_algo(w.N - w.n_decode, w.Hv, w.Dk, w.Dv, 1,
                                                       args.algo),
            "roofline": roof, "kernels": kernels, "gpu_launches": res["launches"],
            "clocks": res["clocks"]}
    if rank == 0 and not args.no_extra:
        extra = {}
        for name in ("decode_b256", "prefill_4k"):
            wx = W.named(name)
            rx = time_workload(wx, dev, max(args.steps, 10), max(args.warmup, 3), args.algo)
            _, rf, kx = roofline_entry(wx, rx["kernel_ms"], peaks)
            extra[name] = {"tokens_per_s": round(wx.T / (rx["ms_per_step"] * 1e-3), 1),
                           "ms_per_step": round(rx["ms_per_step"], 4), "roofline": rf,
                           "kernels": kx}
            del wx
        extra["gated_rmsnorm"] = time_gated_rmsnorm(w, dev, peaks)
        extra["out_norm_routes"] = time_out_norm_routes(w, dev, args.algo)
        extra["kda_decode_b256"] = time_kda_decode(dev, peaks)
        extra["kda_prefill_4k"] = time_kda_prefill(dev, peaks)
        extra["spec_decode_r128x4"] = time_spec_decode(dev, peaks)
        extra["spec_prepare_r128x4"] = time_spec_prepare(dev, peaks)
        extra["packed_decode_b256"] = time_packed_decode(dev, peaks)
        line["extra_workloads"] = extra
    if rank == 0 and not args.no_e2e:
        line["e2e"] = time_e2e(w, dev, max(3, args.steps), 3, args.algo)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        line["cpu_baseline"] = cpu_baseline(w, os.cpu_count() or 1)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
