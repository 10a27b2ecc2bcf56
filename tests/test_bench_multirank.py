"""The multi-process side of bench.py on CPU: two gloo ranks, each timing its
own replica; the job time is the maximum over ranks and the aggregate
throughput counts every rank's tokens."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [120.0, 150.0][rank]
    m = bench.max_over_ranks(elapsed)
    v = bench.aggregate_tokens_per_s(world, 32768, 10, m)
    q.put((rank, m, v))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_two_gloo_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in res:
        assert m == 150.0
        assert v == pytest.approx(2 * 32768 * 10 / 0.150)


def test_single_process_fallbacks():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate_tokens_per_s(1, 100, 4, 2000.0) == pytest.approx(200.0)
