"""The benchmark's multi-rank logic on CPU ranks (gloo, world size 2): the
timed region's result is the slowest rank's time, the job's value counts every
rank's replica, and the reference arm runs on rank 0 alone.  The path has no
exchange step, so this is all the N > 1 path adds."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    local_ms = [120.0, 150.0][rank]
    slowest = bench.max_over_ranks(local_ms, world, "cpu")
    dist.barrier()
    # the reference arm: every rank but 0 returns at once, printing nothing
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    printed = ""
    if rank != 0:
        argv, sys.argv = sys.argv, ["bench.py", "--impl", "reference", "--gpus", str(world)]
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.main()
        sys.argv = argv
        printed = buf.getvalue()
    out.put((rank, slowest, bench.job_throughput(world, 10, slowest), printed))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, printed in res:
        assert slowest == 150.0                  # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * 10 / 0.150)  # both replicas' steps in the job's value
    assert res[1][3] == ""                       # rank 1 ran no reference arm


def test_one_rank_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(42.0, 1, "cpu") == 42.0
    assert bench.job_throughput(1, 100, 500.0) == pytest.approx(200.0)
