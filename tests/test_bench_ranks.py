"""CPU checks of the benchmark's multi-rank path (independent replicas, one per GPU): the
job's time is the slowest rank's, the whole-job value counts every rank's solve, and only
rank 0 runs the reference arm. World size 2 on the gloo backend, 127.0.0.1 rendezvous."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 30.0][rank]
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        out[rank] = (ms, bench.job_seconds_per_solve(ms, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo_world2():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]                       # every rank reports the same job time
    ms, value = res[0]
    assert ms == 30.0                             # the slowest replica sets the clock
    assert value == pytest.approx(30.0 / 1000.0 / 2)   # two solves per step


def test_single_process_is_identity():
    assert bench.max_over_ranks(7.25, None, "cpu") == 7.25
    assert bench.job_seconds_per_solve(100.0, 1) == pytest.approx(0.1)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(workload=1, warmup=1, steps=1, cpu_sample_iters=1, gpus=2))()
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    """The reference arm (the oracle on the host cores) prints one JSON line with the keys
    the harness reads; a bounded sample of the 64 x 64 Laplacian solve keeps it quick."""
    import json
    monkeypatch.setenv("RANK", "0")
    args = type("A", (), dict(workload=1, warmup=1, steps=2, cpu_sample_iters=3, gpus=1))()
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "s" and line["higher_is_better"] is False
    assert line["metric"] == bench.METRIC and line["steps"] == 2 and line["warmup"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["value"] is None or line["value"] > 0
