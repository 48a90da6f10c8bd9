"""The benchmark's multi-rank path (replicas, one process per GPU) on CPU: two gloo ranks
exercise the rendezvous, the barrier and the max-over-ranks timing reduction that bench.py
uses under torchrun, and the whole-job aggregate it prints."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench

    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    # each rank's timed-region seconds differ; every rank must see the max
    t = bench.reduce_max(1.0 + 0.5 * rank, w)
    bench.barrier(w)
    out.put((rank, t))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_and_barrier():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(q.get(timeout=5) for _ in range(world))
    assert got == {0: 1.5, 1: 1.5}


def test_single_rank_path_needs_no_process_group():
    import bench

    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)  # no-op


def test_whole_job_aggregate_uses_all_ranks_units_over_the_slowest_rank():
    import bench

    # 2 ranks x 5 steps x 256 tokens over the slowest rank's 0.5 s
    assert bench.whole_job_rate(world=2, steps=5, units_per_step=256, t_max=0.5) == pytest.approx(5120.0)
