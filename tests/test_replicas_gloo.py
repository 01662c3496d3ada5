"""Replica aggregation of bench.py on CPU: two gloo ranks, barrier, max over ranks.

The layer shards by tokens with no data-path collective, so N GPUs run N
independent replicas; the job time is the slowest rank and the value counts
every rank's tokens.
"""
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


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    own_ms = 100.0 + 50.0 * rank            # rank 1 is the slow replica
    mx = bench.reduce_max(own_ms, world, device="cpu")
    val = bench.whole_job_value(16, 10, mx, world)
    out.put((rank, mx, val))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [150.0, 150.0]
    # 2 ranks x 16 tokens x 10 steps in 0.15 s
    assert all(abs(r[2] - 2 * 16 * 10 / 0.15) < 1e-6 for r in res)


def test_single_rank_is_a_passthrough():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(12.5, 1) == 12.5
    assert bench.whole_job_value(16, 100, 110.0, 1) == pytest.approx(16 * 100 / 0.11)
