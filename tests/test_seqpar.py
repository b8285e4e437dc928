"""Sequence parallelism, host logic on CPU: one sequence cut into segments whose
long memory is handed over by an associative scan of per-segment summaries
(decay A_r, zero-start final state S_r) and whose windows reach back into a
w-token halo.  The fp64 oracle is the engine here, so the segmented result is
compared with the oracle's unsegmented one; the exchange runs in-process and
on gloo ranks (world sizes 2 and 3).  The GPU kernels are exercised by
tests/test_seqpar_gpu.py.  Unmeasured on hardware: every box here has one GPU.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from sliding_window_softmax_gb300.seqpar import (backward_rank, backward_segments, forward_rank,
                                                 forward_segments, segment_plan)


def _inputs(B, H, T, d, m, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, T, d, generator=g, dtype=torch.float64) * d ** -0.25
    k = torch.randn(B, H, T, d, generator=g, dtype=torch.float64) * d ** -0.25
    v = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    la = torch.nn.functional.logsigmoid(torch.randn(B, H, T, m, generator=g, dtype=torch.float64) + 2.0)
    dout = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    return q, k, v, la, dout


def test_segment_plan_covers_the_sequence():
    for T, n, w in [(10, 1, 3), (100, 3, 7), (101, 4, 0), (64, 8, 100)]:
        plan = segment_plan(T, n, w)
        assert plan[0].a == 0 and plan[-1].b == T
        for s, t in zip(plan, plan[1:]):
            assert s.b == t.a
        for s in plan:
            assert s.lo == max(0, s.a - w) and s.keep == s.a - s.lo and s.b > s.a
    with pytest.raises(ValueError):
        segment_plan(3, 4, 1)


@pytest.mark.parametrize("n,w", [(2, 5), (3, 7), (4, 0), (3, 30)])
def test_segments_in_process_equal_the_whole_sequence(n, w):
    from seqpar_engines import oracle_engine

    q, k, v, la, dout = _inputs(1, 2, 61, 8, 3, seed=700 + n + w)
    eng = oracle_engine()
    o, lse, ctx = forward_segments(q, k, v, la, w, n, engine=eng)
    ro, rlse = oracle.forward(q, k, v, la, w)
    assert np.abs(o.numpy() - ro).max() <= 1e-10
    assert np.abs(lse.numpy() - rlse).max() <= 1e-10
    g = backward_segments(ctx, dout, engine=eng)
    rg = oracle.backward(q, k, v, la, dout, w)
    for name, a, b in zip(("dq", "dk", "dv", "dla"), g, rg):
        assert np.abs(a.numpy() - b).max() <= 1e-9 * max(1.0, np.abs(b).max()), name


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, w, q_out):
    import sys

    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import torch.distributed as dist

    from seqpar_engines import oracle_engine

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, la, dout = _inputs(1, 2, 70, 8, 3, seed=800 + world)
        s = segment_plan(70, world, w)[rank]
        sl = slice(s.a, s.b)
        eng = oracle_engine()
        o, lse, ctx = forward_rank(q[:, :, sl], k[:, :, sl], v[:, :, sl], la[:, :, sl], w, engine=eng)
        g = backward_rank(ctx, dout[:, :, sl], engine=eng)
        q_out.put((rank, s.a, s.b, o.numpy(), lse.numpy(), [x.numpy() for x in g]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,w", [(2, 9), (3, 12)])
def test_segments_on_gloo_ranks_equal_the_whole_sequence(world, w):
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, w, q_out)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q_out.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    q, k, v, la, dout = _inputs(1, 2, 70, 8, 3, seed=800 + world)
    ro, rlse = oracle.forward(q, k, v, la, w)
    rg = oracle.backward(q, k, v, la, dout, w)
    for rank, a, b, o, lse, g in res:
        assert np.abs(o - ro[:, :, a:b]).max() <= 1e-10, rank
        assert np.abs(lse - rlse[:, :, a:b]).max() <= 1e-10, rank
        for name, x, r in zip(("dq", "dk", "dv", "dla"), g, rg):
            assert np.abs(x - r[:, :, a:b]).max() <= 1e-9 * max(1.0, np.abs(r).max()), (rank, name)
