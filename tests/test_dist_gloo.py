"""Multi-rank host logic of the benchmark on the CPU (gloo, 2 ranks): every
rank owns its own sequences (weak scaling, no collective on the data path)
and the job time is the maximum over ranks."""
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
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.reduce_max(1.0 + rank * 2.5, dist)
        shard = bench.shard_sequences(34, rank)
        gathered = [None] * world
        dist.all_gather_object(gathered, shard)
        q.put((rank, t, gathered))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_disjoint_shards():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, gathered in res:
        assert t == pytest.approx(3.5)
        flat = [s for shard in gathered for s in shard]
        assert len(flat) == 68 and len(set(flat)) == 68


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_max(4.25, None) == 4.25
    assert bench.shard_sequences(5, 0) == [0, 1, 2, 3, 4]
