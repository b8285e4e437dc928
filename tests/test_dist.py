"""Multi-rank host logic on CPU (gloo, world_size 2): head partition and the
max-over-ranks timing reduction used by bench.py.  No GPU involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from sliding_window_softmax_gb300.dist import head_partition, heads_of, max_over_ranks


def test_partition_covers_every_head_once():
    for B, H in [(1, 1), (4, 16), (3, 5), (2, 7)]:
        for world in (1, 2, 3, 8):
            got = []
            for r in range(world):
                s, e = head_partition(B, H, world, r)
                assert 0 <= e - s <= (B * H + world - 1) // world
                got += heads_of(B, H, world, r)
            assert sorted(got) == [(b, h) for b in range(B) for h in range(H)]
    with pytest.raises(ValueError):
        head_partition(2, 2, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = max_over_ranks([1.0 + rank, 10.0 - rank])
        s, e = head_partition(4, 16, world, rank)
        counts = torch.tensor([e - s])
        dist.all_reduce(counts)
        q.put((rank, mx, int(counts.item())))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
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
    for rank, mx, total in res:
        assert mx == [2.0, 10.0]
        assert total == 64


def test_max_over_ranks_without_process_group():
    assert max_over_ranks([3.0, 1.5]) == [3.0, 1.5]
