"""Host logic of multi-GPU runs, on CPU with the gloo backend (world size 2).

The method shards by independent (b, h) heads, so a multi-GPU run has no
data-path collective: every rank runs its own workload and the ranks only agree
on the slowest rank's time. These tests check that reduction and the whole-job
throughput built from it, with real processes on 127.0.0.1.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(ws)
        slowest = bench.max_over_ranks(times[rank], ws, device="cpu")
        results[rank] = (slowest, bench.aggregate_tokens_per_s(32768, slowest, ws))
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_slowest_time_and_aggregate():
    world = 2
    times = [1.25, 3.5]  # ms per step measured on each rank
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        slowest, tps = results[r]
        assert slowest == 3.5
        assert tps == pytest.approx(2 * 32768 / 3.5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.0, 1) == 2.0
    assert bench.aggregate_tokens_per_s(1000, 2.0, 1) == pytest.approx(5e5)
