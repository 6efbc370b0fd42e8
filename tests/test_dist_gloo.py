"""The multi-replica path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The decode step does not shard (every rank runs its own replica of the layer
on its own GPU, no collective on the data path); the only cross-rank steps
are the barriers around the timed loop, the max of the per-rank times and
the whole-job aggregate.  These run here with the gloo backend.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import io
    import contextlib

    import torch.distributed as dist

    import bench

    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.barrier()
    # per-rank times differ; the job ends with the slowest rank
    local_ms = 10.0 + 5.0 * rank
    ms_max = bench.max_over_ranks(local_ms)
    us = bench.whole_job_us_per_decode(ms_max, steps=100, world=w)
    # the reference arm prints on rank 0 only; other ranks do no work
    buf = io.StringIO()
    if rank != 0:
        with contextlib.redirect_stdout(buf):
            bench.run_reference(bench.parse_args(["--impl", "reference"]))
    bench.barrier()
    out.put((rank, ms_max, us, buf.getvalue()))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = dict((r, (m, u, o)) for r, m, u, o in results)
    for r in range(world):
        ms_max, us, printed = by_rank[r]
        assert ms_max == pytest.approx(15.0)  # max over ranks, same on every rank
        # 15 ms for 100 steps on each of 2 replicas: 75 us per decode, job-wide
        assert us == pytest.approx(75.0)
    assert by_rank[1][2] == ""


def test_single_process_helpers_without_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_us_per_decode(2.0, steps=10, world=1) == pytest.approx(200.0)
    bench.barrier()  # no process group: a no-op
