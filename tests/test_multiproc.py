"""Host logic of the multi-GPU bench path on CPU: two gloo ranks shard the
independent (batch, head) units with no data-path collective and reduce only
their step times (max over ranks)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lo, hi = bench.shard_units(96, world, rank)
        my_ms = 1.0 + rank  # rank 1 is the slow one
        t = torch.tensor([my_ms], dtype=torch.float64)
        gathered = [torch.zeros_like(t) for _ in range(world)]
        dist.all_gather(gathered, t)
        agg = bench.aggregate([float(x) for x in gathered], 1e12, 1000)
        q.put((rank, lo, hi, agg))
    finally:
        dist.destroy_process_group()


def test_two_rank_sharding_and_max_timing():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert [(r[1], r[2]) for r in results] == [(0, 48), (48, 96)]
    for _, _, _, agg in results:
        assert agg["ms_per_step"] == 2.0
        assert agg["tflops"] == pytest.approx(2 * 1e12 / 2e-3 / 1e12)


def test_shard_units_cover_exactly():
    for n in (1, 7, 96, 100):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_units(n, world, r) for r in range(world)]
            covered = [i for lo, hi in spans for i in range(lo, hi)]
            assert covered == list(range(n))
