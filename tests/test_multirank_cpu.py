"""Multi-process host logic on CPU (gloo, world size 2): sequence sharding
covers every row exactly once without splitting a verify group, and the step
time reduces to the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sparse_attention_mla_dsa_gb300 import shard


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, rows, rows_per_seq, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = shard.shard_rows(rows, rows_per_seq, rank, world)
        got = [None] * world
        dist.all_gather_object(got, list(mine))
        t = shard.max_over_ranks(1.5 + rank)     # rank r reports 1.5 + r ms
        q.put((rank, got, t))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("rows,rows_per_seq", [(32, 4), (33, 1), (4, 4)])
def test_sharding_and_max_timing_gloo_ws2(rows, rows_per_seq):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, rows, rows_per_seq, q))
             for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, t in results:
        flat = [r for part in got for r in part]
        assert flat == list(range(rows))                     # every row once, in order
        for part in got:
            assert len(part) % rows_per_seq == 0             # verify groups stay whole
        assert t == 1.5 + (world - 1)                        # max over ranks


def test_shard_groups_balanced():
    sizes = [len(shard.shard_groups(10, r, 4)) for r in range(4)]
    assert sizes == [3, 3, 2, 2]
    with pytest.raises(ValueError):
        shard.shard_groups(10, 4, 4)
    with pytest.raises(ValueError):
        shard.shard_rows(10, 4, 0, 2)
