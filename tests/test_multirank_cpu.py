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


def _norm_worker(rank, world, port, q):
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle
    import rollout_consistent_vocab_gb300 as pkg
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = np.random.default_rng(3).standard_normal(10001).astype(np.float32) * 1e-2
    mine = np.array_split(x, world)[rank]
    bins = torch.from_numpy(oracle.sqnorm_bins(mine, "f32").view(np.int64).copy())
    pkg.reduce_bins_(bins)
    q.put((rank, oracle.norm_finalize(bins.numpy().view(np.uint64))))
    dist.barrier()
    dist.destroy_process_group()


def test_norm_bins_distributed_reduction_gloo():
    """The gradient norm's distributed reduction (an integer all-reduce of the
    bins) over two ranks gives the single-rank result exactly."""
    import numpy as np
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_norm_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x = np.random.default_rng(3).standard_normal(10001).astype(np.float32) * 1e-2
    want = oracle.grad_norm(x, "f32")
    assert [r[1] for r in res] == [want, want]


def test_cpu_baseline_one_process_per_core():
    """bench.py's all-core CPU baseline: every core's process reports rows."""
    import numpy as np
    import torch
    import bench
    from rollout_consistent_vocab_gb300 import workloads as W
    wl = W.workload_c2(device="cpu", T=4)
    bits = wl.logits.view(torch.int16).numpy().view(np.uint16)
    rbits = wl.ref_logits.view(torch.int16).numpy().view(np.uint16)
    tg = W.structural_targets(4, wl.hot, wl.hot_n, seed=2).numpy()
    rate, rows, secs, ncores = bench.cpu_oracle_rate_all_cores(bits, rbits, tg, 1.0)
    assert ncores >= 1 and rows >= ncores and secs >= 1.0 and rate == rows / secs


def test_reference_arm_prints_one_complete_line(capsys):
    """bench.py --impl reference on rank 0: one JSON line with the contract's keys."""
    import json
    import bench

    class A:
        steps, warmup, gpus = 1, 0, 1
    bench.run_reference(A, rank=0, world=1)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_bench_parity_object_from_the_cpu_leg():
    """bench.py's parity object: the single-core oracle leg's results against
    outputs for the same rows; exact outputs pass, a planted deviation counts."""
    import numpy as np
    import torch
    import bench
    from rollout_consistent_vocab_gb300 import workloads as W
    wl = W.workload_c2(device="cpu", T=3)
    bits = wl.logits.view(torch.int16).numpy().view(np.uint16)
    rbits = wl.ref_logits.view(torch.int16).numpy().view(np.uint16)
    tg = W.structural_targets(3, wl.hot, wl.hot_n, seed=2).numpy()
    rate, n, secs, res = bench.cpu_oracle_rate(bits, rbits, tg, 60.0)
    assert n == 3 and len(res) == 3
    full = np.array([r.full for r, _ in res], np.float32)
    restr = np.array([r.restr for r, _ in res], np.float32)
    sup = np.array([r.support for r, _ in res], np.int32)
    fref = np.array([f for _, f in res], np.float32)
    kl = full - fref
    d = bench.parity_summary(res, full, restr, sup, fref, kl)
    assert d["pass"] and d["rows"] == 3 and d["rows_over_tol"] == 0 and d["support_differs"] == 0
    full[1] += 1e-3
    d = bench.parity_summary(res, full, restr, sup, fref, kl)
    assert not d["pass"] and d["rows_over_tol"] >= 1
