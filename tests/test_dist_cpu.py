"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2):
rows are independent, so ranks run replicas and only the elapsed time is
reduced (max over ranks); no data-path collective exists."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, _ = bench.dist_env()
    assert (r, w) == (rank, world)
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    got = bench.max_over_ranks(ms, torch.device("cpu"))
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_job_throughput_is_weak_scaling():
    import bench
    one = bench.job_gbs(1_000_000, 10, 1, 2.0)
    two = bench.job_gbs(1_000_000, 10, 2, 2.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(1e7 / 2e-3 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
