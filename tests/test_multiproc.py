"""Host logic of the multi-GPU bench path on CPU: two gloo ranks each draw
their own batch (their own seeds; no data-path collective) and reduce only
their step times (max over ranks)."""

import dataclasses
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
        from block_sparse_long_bigbird_gb300.workloads import WORKLOADS
        wl = WORKLOADS["bigbird_bf16_n4096"]
        # each rank's batch comes from its own seeds: no rank needs another's data
        q_first = bench.make_inputs(dataclasses.replace(wl, B=1, H=1, n=128), rank)["Q"][0, 0, 0, :4].float()
        my_ms = 1.0 + rank  # rank 1 is the slow one
        t = torch.tensor([my_ms], dtype=torch.float64)
        gathered = [torch.zeros_like(t) for _ in range(world)]
        dist.all_gather(gathered, t)
        agg = bench.aggregate([float(x) for x in gathered], 1e12, 1000)
        q.put((rank, bench.rank_seed_offset(rank), q_first.tolist(), agg))
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
    assert [r[1] for r in results] == [0, 100]
    assert results[0][2] != results[1][2], "ranks must draw different batches"
    for _, _, _, agg in results:
        assert agg["ms_per_step"] == 2.0
        assert agg["tflops"] == pytest.approx(2 * 1e12 / 2e-3 / 1e12)
