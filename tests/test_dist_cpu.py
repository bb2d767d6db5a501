"""bench.py's multi-process plumbing on CPU: two gloo ranks, barrier and max-over-ranks timing."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    ms = bench.max_over_ranks(10.0 * (rank + 1), w, "cpu")
    out[rank] = ms
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    import bench

    class A:
        steps, warmup, workload = 1, 0, bench.DEFAULT_WORKLOAD

    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "make_pool", lambda cores: called.append(cores))
    assert bench.run_reference(A()) is None
    assert called == []
