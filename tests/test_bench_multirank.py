"""The multi-GPU path of bench.py on the CPU: replicas with no data-path
collective, two gloo ranks.  Each rank's inputs are its own shard (other
seeds, same shapes); the job's time is the slowest rank's; the whole-job
rate counts every rank's positions."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 7.0 * rank  # this rank's elapsed ms
        slowest = bench.max_over_ranks(mine, torch.device("cpu"))
        tdist.barrier()
        q.put((rank, slowest))
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == {0: 17.0, 1: 17.0}


def test_job_rate_counts_every_rank():
    per = bench.positions_per_step()
    assert bench.job_rate(per, 1, 10, 2.0) == pytest.approx(per * 10 / 2e-3)
    assert bench.job_rate(per, 4, 10, 2.0) == pytest.approx(4 * bench.job_rate(per, 1, 10, 2.0))


def test_rank_shards_differ_with_equal_shapes():
    # a small stand-in of the benchmark workload (the generator takes the shape)
    import workloads as W
    a = W.config3(seed=3, B=4, k=2, V=512)
    b = W.config3(seed=4, B=4, k=2, V=512)
    assert a.target.shape == b.target.shape and a.tokens.shape == b.tokens.shape
    assert not np.array_equal(a.target, b.target) and not np.array_equal(a.uniforms, b.uniforms)
