"""The N > 1 path of bench.py (independent replicas, max-over-ranks timing)
on CPU: two gloo ranks."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")  # rank 1 is the slow replica
    dist.barrier()
    q.put((rank, slowest, bench.job_rate(world, 256 * 3, slowest / 1000.0)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    mp = pytest.importorskip("torch.multiprocessing")
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [15.0, 15.0]
    # whole-job tokens/s: both replicas' tokens over the slowest replica's time
    assert out[0][2] == pytest.approx(2 * 768 / 0.015)
