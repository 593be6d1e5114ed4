"""The N > 1 bench path on CPU: two gloo ranks (replicas, no data-path
collective). Whole-job throughput is the units of all ranks over the slowest
rank's time; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dev = torch.device("cpu")
        bench.barrier(dev)
        # rank r pretends its timed region took r + 1 seconds for 10 (r + 1) units
        el, units = bench.aggregate_ranks(float(rank + 1), 10.0 * (rank + 1), dev)
        out[rank] = (el, units, bench.dist_env())
        bench.barrier(dev)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_summed_units():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        el, units, env = out[r]
        assert el == 2.0                  # the slowest rank's time
        assert units == 30.0              # 10 + 20 units over both ranks
        assert env == (world, r, r)


def test_aggregate_without_process_group_is_identity():
    assert bench.aggregate_ranks(1.5, 7.0, torch.device("cpu")) == (1.5, 7.0)


def test_every_rank_runs_the_same_workload():
    # replicas: no rank-dependent slicing of the problems
    assert bench.WORKLOADS["decode-7b"] == [(M, K, N, 128, False) for M in (1, 4, 16)
                                            for (K, N) in bench.DECODE_SHAPES]


def test_reference_arm_is_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    called = []
    monkeypatch.setattr(bench, "run_reference", lambda *a, **k: called.append(1))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    bench.main()
    assert called == [] and capsys.readouterr().out == ""


def test_reference_arm_line_on_one_rank(monkeypatch, capsys):
    """At N = 1 the reference arm (the CPU oracle on a bounded sample) prints
    one JSON line with the bench contract's keys, on the native arm's metric
    and workload, and its cpu_baseline and e2e values equal to the line's."""
    import json
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3"])
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["unit"] == "TFLOP/s"
    assert d["config"]["workload"] == bench.DEFAULT_WORKLOAD and d["data"] == "synthetic"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
