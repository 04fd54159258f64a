"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): ranks use
disjoint seeds, the job time is the slowest rank's, throughput counts every
rank's rows, and only rank 0 runs the CPU reference arm."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank
    slowest = bench.max_over_ranks(local_ms, torch.device("cpu"))
    seeds = [None] * world
    dist.all_gather_object(seeds, bench.rank_seed(2, rank))
    q.put((rank, slowest, bench.throughput(world, 8192, 4, slowest), seeds))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, thr, seeds in res:
        assert slowest == 15.0
        assert thr == pytest.approx(2 * 8192 * 4 / 0.015)
        assert len(set(seeds)) == 2


def test_reference_arm_other_ranks_exit_silently(capsys):
    import bench

    class A:
        steps, warmup, gpus = 1, 0, 2
    assert bench.run_reference(A, rank=1, world=2) is None
    assert capsys.readouterr().out == ""
