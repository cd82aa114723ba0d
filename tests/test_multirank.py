"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The path shards over independent blocks (replicas of the workload, no data
exchange), so the only multi-rank logic is the timing: each timing is the
maximum over the ranks, and the whole job's µs per pass divides that time by
the passes all ranks ran.  The reference arm runs on rank 0 alone."""

import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        # rank r measured (10 + r, 5 - r): the maxima are (10 + world - 1, 5)
        got = bench.max_over_ranks([10.0 + rank, 5.0 - rank], world, torch.device("cpu"))
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_timings_are_max_over_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    for r in range(world):
        assert out[r] == [10.0 + world - 1, 5.0]


def test_whole_job_value_counts_every_rank():
    import bench

    # 200 passes per rank in 18,400 us on each of 4 ranks: 800 passes, 23 us each
    assert bench.whole_job_per_pass(18400.0, 200, 4) == pytest.approx(23.0)
    assert bench.whole_job_per_pass(18400.0, 200, 1) == pytest.approx(92.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1"])
    called = []
    monkeypatch.setattr(bench, "run_reference", lambda args, world: called.append(world))
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main()  # rank 1: returns at once, prints nothing
    assert called == [] and buf.getvalue() == ""
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_RANK", "0")
    bench.main()
    assert called == [2]


def test_config_names_replicas_above_one_rank():
    import bench

    assert bench.workload_config(1)["parallelism"] == "single GPU"
    assert bench.workload_config(4)["parallelism"] == "replicas"
    assert bench.workload_config(4)["workload"] == bench.workload_config(1)["workload"]
