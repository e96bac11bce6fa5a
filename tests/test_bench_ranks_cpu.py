"""Multi-rank host logic of bench.py on CPU: two gloo ranks (replicas), the
job's step time is the slowest rank's, and the job's throughput counts every
rank's bytes."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        ms_local = [0.25, 0.40][rank]   # rank 1 is the slow one
        ms = bench.max_over_ranks(torch, dist, ms_local, "cpu")
        gbs = bench.job_throughput(world, 1_000_000, ms)
        q.put((rank, ms, gbs))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, gbs in got:
        assert ms == pytest.approx(0.40)
        assert gbs == pytest.approx(2 * 1_000_000 / 0.40e-3 / 1e9)


def test_job_throughput_single_rank():
    bench = _bench()
    assert bench.job_throughput(1, 514_569_216, 0.25) == pytest.approx(514_569_216 / 0.25e-3 / 1e9)
