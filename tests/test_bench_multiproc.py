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


def test_kernel_hash_follows_code_not_comments():
    # bench.py reports the ncu traffic of profiles/ only while the kernel's code
    # is the one that was captured: comment edits keep the hash, code edits change it.
    sys.path.insert(0, ROOT)
    import bench
    src = {f: open(os.path.join(ROOT, f)).read() for f in bench.KERNEL_SOURCES}
    h0 = bench.kernel_source_hash(lambda f: src[f])
    assert h0 == bench.kernel_source_hash()
    f = bench.KERNEL_SOURCES[0]
    commented = dict(src)
    commented[f] = "// a new comment line\n" + src[f].replace("\n", "  // trailing note\n", 1) + "\n/* block\n   comment */\n"
    assert bench.kernel_source_hash(lambda g: commented[g]) == h0
    changed = dict(src)
    changed[f] = src[f] + "\nconstexpr int unused_probe = 1;\n"
    assert bench.kernel_source_hash(lambda g: changed[g]) != h0
