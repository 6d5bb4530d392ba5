"""The N > 1 host path of bench.py on CPU: two gloo ranks, each a replica of the workload.

The layer partitions into independent (sequence, head) units with no exchange step, so
N GPUs run N replicas: the only cross-rank operations are the barrier and the max of the
per-rank step times, and the whole-job rate is N x units / slowest time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    torch.cuda.is_available = lambda: False  # CPU ranks over gloo, also on a machine with a GPU
    d, r, w, local = bench._dist()
    try:
        assert (r, w, local) == (rank, world, rank)
        bench._barrier(d)
        step_ms = 1.0 + rank  # rank 1 is the slow one
        ms_max = bench._max_over_ranks(d, step_ms)
        q.put((rank, ms_max, bench.weak_scaling_rate(w, 10240, ms_max)))
    finally:
        d.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms_max, rate in got:
        assert ms_max == 2.0  # the slowest rank's time, on every rank
        assert rate == pytest.approx(2 * 10240 / 2.0e-3)


def test_single_rank_needs_no_process_group():
    assert bench._dist()[0] is None or os.environ.get("WORLD_SIZE", "1") != "1"
    assert bench._max_over_ranks(None, 3.5) == 3.5
    assert bench.weak_scaling_rate(1, 1000, 2.0) == pytest.approx(5e5)
