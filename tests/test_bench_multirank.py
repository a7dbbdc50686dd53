"""bench.py's multi-rank path on CPU: two gloo ranks, slowest-rank timing and
whole-job throughput (replicas: every rank runs the full workload)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, rank, world)
        slowest = bench.max_over_ranks(0.010 + 0.005 * rank)  # rank 1 is slower
        gbs = bench.replica_throughput(134217728, 10, world, slowest)
        dist.barrier()
        q.put((rank, slowest, gbs))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, gbs in got:
        assert slowest == pytest.approx(0.015)
        assert gbs == pytest.approx(2 * 134217728 * 10 / 0.015 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.replica_throughput(100, 2, 1, 1e-9) == pytest.approx(200.0)
