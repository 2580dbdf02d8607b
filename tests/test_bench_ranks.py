"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks agree on the
slowest rank's step time and on the whole-job throughput, and only rank 0 of
the reference arm prints.  The layer runs as independent replicas (one per
GPU, no collective on the data path), so the aggregation is the only
multi-rank logic."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.rank_info()
        ms = 1.0 + 0.5 * rank           # rank 1 is the slow replica
        slow = bench.slowest_rank_ms(ms, dist, torch.device("cpu"))
        value = bench.whole_job_value(8704, got_ws, slow)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
            json.dump({"ws": got_ws, "rank": got_rank, "local": got_local, "slow": slow,
                       "value": value}, fh)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step(tmp_path):
    ws, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(ws, port, str(tmp_path)), nprocs=ws, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(ws)]
    for r, d in enumerate(res):
        assert (d["ws"], d["rank"], d["local"]) == (ws, r, r)
        assert d["slow"] == pytest.approx(1.5)
        assert d["value"] == pytest.approx(8704 * 2 / 1.5e-3)


def test_single_rank_needs_no_collective():
    assert bench.slowest_rank_ms(2.5, None, None) == 2.5
    assert bench.whole_job_value(1000, 1, 2.0) == pytest.approx(5e5)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_times_whole_oracle_steps(monkeypatch, capsys):
    """The reference arm runs W + K whole oracle steps of the workload (no
    extrapolation): its timed steps fit inside the wall time of the call, and
    it prints the same config object as the GPU arm."""
    import time
    from gated_delta_rule_44_gb300 import workloads as W
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--workload",
                                      "tiny_f32", "--steps", "3", "--warmup", "1"])
    t0 = time.perf_counter()
    assert bench.main() == 0
    wall = time.perf_counter() - t0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    w = W.named("tiny_f32")
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 1
    assert line["config"] == bench.workload_config(w, 1)
    assert line["ms_per_step"] * 3 / 1e3 <= wall
    assert line["value"] == pytest.approx(w.T / (line["ms_per_step"] / 1e3), rel=1e-3)
    assert "no extrapolation" in line["cpu_baseline"]["sample"]
