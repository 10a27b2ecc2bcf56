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


def test_reference_arm_prints_the_contract_line():
    """The reference arm times the oracle on the host cores and prints one JSON
    line with the contract's keys (small sample so the test stays fast)."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "0", "--ref-sample-tokens", "256"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["higher_is_better"] is True and line["config"]["workload"] == "tiny"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
