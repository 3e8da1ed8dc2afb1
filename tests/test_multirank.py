"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Every GPU runs its own replica of the benchmark step (the layer does not shard across GPUs
here), so the only cross-rank logic is the timing: the job's time is the slowest rank's, and the
job's rate counts every rank's units.  The reference arm runs on rank 0 only.
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
