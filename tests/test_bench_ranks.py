"""Host logic of the bench's multi-GPU path, on the CPU with gloo.

With N ranks the bench runs N independent replicas (one megabatch each, no
collective on the data path).  Each rank times its own region; the line
reports the slowest rank's time (an all-reduce MAX over the ranks) and the
whole-job time per megabatch, i.e. that time divided by N.  The reference
arm runs on rank 0 only; the other ranks exit without work.
"""
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench

TIMES = [3.0, 7.5]


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(TIMES[rank], world, torch.device("cpu"))
        q.put((rank, got, bench.job_value(got, world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_job_value_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 7.5, 3.75), (1, 7.5, 3.75)]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.25, 1, None) == 4.25
    assert bench.job_value(4.25, 1) == 4.25


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        workload = "gpt-small-megabatch"
        steps = 1
        warmup = 0
    assert bench.run_reference(Args(), 1, 2) is None
    assert capsys.readouterr().out == ""
