"""The N > 1 paths on CPU: two gloo ranks on 127.0.0.1.

- bench.py's timing: the job's time is the slowest rank's, and the job's rate counts every
  rank's units; the reference arm runs on rank 0 only.
- The column-parallel split (w4a16_group_wise_gb300.shard): the ranks' column ranges partition
  [0, N) on 64-column boundaries, and gathering every rank's columns of y rebuilds y whole.
"""
import argparse
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
    rate = bench.whole_job_rate(1.0e6, world, ms)
    ref = bench.run_reference(argparse.Namespace(steps=1, warmup=0), rank, world) if rank > 0 else "skipped"
    dist.barrier()
    q.put((rank, ms, rate, ref))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_units():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate, ref in out:
        assert ms == 15.0                      # the slower rank's 15 ms, on every rank
        assert rate == pytest.approx(2.0e6 / 15e-3)
        if rank > 0:
            assert ref is None                 # only rank 0 runs the reference arm


def test_one_rank_is_unchanged():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_rate(7.0, 1, 2.0) == pytest.approx(3500.0)


def _shard_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from w4a16_group_wise_gb300 import shard
    out = {}
    for N in (13312, 3072, 80, 131072, 2048 + 8):
        mine = shard.column_slices(N, world)[rank]
        every = [None] * world
        dist.all_gather_object(every, mine)
        out[N] = every
    # gather of y: every rank fills its columns of a known y; the gathered y is y whole
    M, N = 3, 200
    part = shard.ColumnParallelLinear.__new__(shard.ColumnParallelLinear)
    part.slices, part.world = shard.column_slices(N, world), world
    n0, n1 = part.slices[rank]
    y_full = torch.arange(M * N, dtype=torch.float32).reshape(M, N)
    y_gathered = part.gather(y_full[:, n0:n1].contiguous())
    dist.barrier()
    q.put((rank, out, bool(torch.equal(y_gathered, y_full))))
    dist.destroy_process_group()


def test_two_ranks_split_the_columns_and_gather_y():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == res[1][1]                   # both ranks see the same partition
    for N, slices in res[0][1].items():
        assert slices[0][0] == 0 and slices[-1][1] == N
        for (a0, a1), (b0, b1) in zip(slices, slices[1:]):
            assert a1 == b0                          # contiguous, disjoint
        for n0, n1 in slices:
            assert n0 % 64 == 0 and n0 <= n1        # n-block aligned starts
            assert n1 == N or n1 % 64 == 0          # only the last end is ragged
        widths = [n1 - n0 for n0, n1 in slices]
        assert max(widths) - min(widths) <= 64      # balanced to one n-block
    assert res[0][1][80] == [(0, 64), (64, 80)]     # the 64 + 16 layer: the tail on the last rank
    assert all(ok for _, _, ok in res)


def test_column_slices_edge_cases():
    import sys
    sys.path.insert(0, ROOT)
    from w4a16_group_wise_gb300 import shard
    assert shard.column_slices(80, 4) == [(0, 0), (0, 0), (0, 64), (64, 80)]   # more ranks than n-blocks
    assert shard.column_slices(64, 1) == [(0, 64)]
    assert shard.column_slices(13312, 8) == [(1664 * r, 1664 * (r + 1)) for r in range(8)]
    assert shard.column_slices(2056, 2) == [(0, 1024), (1024, 2056)]
    with pytest.raises(ValueError):
        shard.column_slices(0, 2)


def test_timed_graphs_span_more_than_l2():
    """bench.py's one-shape timing graphs cycle through at least L2_SPAN bytes of weights (more than
    the 129 MB L2): the buffers given first, then copies of them in turn, each in memory of its own."""
    import torch
    import bench
    assert bench.L2_SPAN > 129e6
    base = [torch.full((3268864,), i, dtype=torch.uint8) for i in range(8)]  # eight q_k_v-sized buffers
    bufs = bench.over_l2(base)
    total = sum(b.numel() * b.element_size() for b in bufs)
    assert total >= bench.L2_SPAN and total - bufs[-1].numel() < bench.L2_SPAN  # no copy beyond the span
    assert len(bufs) == 49 and all(a is b for a, b in zip(bufs, base))
    assert len({b.data_ptr() for b in bufs}) == len(bufs)
    assert all(torch.equal(bufs[i], base[i % 8]) for i in range(len(bufs)))
