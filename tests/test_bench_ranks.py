"""bench.py's multi-rank host logic on CPU with two gloo ranks: every rank runs a replica of
the workload, the job's time is the slowest rank's, and the reported rate counts the units of
all ranks.  The reference arm does its work on rank 0 only."""
import math
import socket
import types

import torch.multiprocessing as mp

import bench
from tests.dist_worker import bench_ranks


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_report_the_slowest_time_and_the_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=bench_ranks, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, rate in got:
        assert ms == 15.0
        assert math.isclose(rate, 2 * 16384 / 0.015)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert math.isclose(bench.job_rate(1, 1000, 2.0), 500000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = types.SimpleNamespace(workload="tiny", steps=1, warmup=0, ref_tokens=8)
    assert bench.run_reference(args, rank=1, world=2) is None
    assert capsys.readouterr().out == ""
