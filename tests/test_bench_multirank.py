"""The replica path of bench.py (one process per GPU, launched by torchrun)
on CPU: two gloo ranks check the slowest-rank time reduction and the
whole-job aggregation, and that only rank 0 of the reference arm prints."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [0.4, 0.7][rank]                       # rank 1 is the slow one
    bench.barrier(world)
    slowest = bench.max_over_ranks(ms, world, torch.device("cpu"))
    value = bench.job_gbs(2 * 2 ** 30, world, slowest)
    w, r, l = bench.dist_setup(None)
    q.put((rank, slowest, value, (w, r, l)))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, env in res:
        assert slowest == 0.7                   # MAX over ranks
        assert abs(value - 2 * 2 * 2 ** 30 / 0.7e-3 / 1e9) < 1e-9   # all ranks' bytes / slowest time
        assert env == (world, rank, rank)


def test_reference_arm_prints_only_on_rank_0(capsys):
    import bench

    class A:  # argparse stand-in
        workload, batch, steps, warmup = 1, 0, 1, 0
    bench.run_reference(A(), world=2, rank=1)
    assert capsys.readouterr().out == ""
