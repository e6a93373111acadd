"""Multi-rank host logic of bench.py on CPU: two gloo ranks with different
elapsed times; the whole-job figure takes the slowest rank and counts every
rank's units (weak scaling, no data-path collective)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        elapsed = 100.0 + 50.0 * rank            # rank 1 is the slow one
        ms, value = bench.combine_ranks(elapsed, units_per_step=1000.0,
                                        steps=10, world=world)
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_combine_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 150.0                       # max over ranks
        assert abs(value - 1000.0 * 10 * 2 / 0.150) < 1e-6 * value


def test_combine_ranks_single():
    import bench
    ms, value = bench.combine_ranks(200.0, 5.0, 4, 1)
    assert ms == 200.0 and abs(value - 5.0 * 4 / 0.2) < 1e-9
