"""The bench's multi-rank timing on CPU: two gloo ranks (127.0.0.1) agree on
the slowest rank's time and on the whole-job throughput, and a single
process (no group) keeps its own value.  No GPU is involved: this is the
host-side logic a torchrun launch of bench.py uses for N > 1 replicas."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        ws, r, local = bench.dist_env()
        ms = bench.max_over_ranks(1.5 + rank, "cpu")    # rank 1 is the slower one
        rate = bench.job_rate(64.0, ws, ms)
        dist.barrier()
        q.put((r, ws, local, ms, rate))
    finally:
        dist.destroy_process_group()


def test_single_process_keeps_its_value():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [g[0] for g in got] == [0, 1]
    for r, ws, local, ms, rate in got:
        assert ws == 2 and local == r
        assert ms == 2.5
        assert rate == pytest.approx(64.0 * 2 / 2.5e-3)
    assert all(p.exitcode == 0 for p in procs)
