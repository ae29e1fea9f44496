"""The benchmark's multi-rank path (one process per GPU, weak scaling, max of
the ranks' times) on CPU with the gloo backend and two ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        my_ms = 10.0 + 5.0 * rank  # the slower rank decides
        worst = bench.max_over_ranks(my_ms)
        bench.barrier()
        q.put((r, lr, w, worst, bench.aggregate_throughput(4096, w, worst / 1e3)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_weak_scaling_aggregation_over_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for r, (rank, lr, w, worst, tput) in enumerate(got):
        assert rank == r and lr == r and w == world
        assert worst == 15.0
        assert tput == pytest.approx(4096 * world / 0.015)


def test_single_process_defaults(monkeypatch):
    import bench
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 0, 1)
    assert bench.max_over_ranks(3.5) == 3.5
