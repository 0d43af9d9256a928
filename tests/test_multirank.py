"""Host logic of the benchmark's N-rank runs, on CPU with the gloo backend.

The path shards by unit with no data-path collective; across ranks the
benchmark only (1) gives each rank its own seeded inputs and (2) takes the
slowest rank's time for the whole-job rate.  Two gloo ranks check both.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    import workloads as W
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        r, wsz, local = bench.dist_env()
        t = bench.max_over_ranks(1.5 + rank, wsz, "cpu")
        w = W.WORKLOADS[1]
        q.put((r, wsz, local, t, bench.whole_job_rate(wsz, 100, t), bench.rank_seed(w, r)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_seeds():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [g[0] for g in got] == [0, 1] and all(g[1] == world for g in got)
    assert all(g[3] == 2.5 for g in got)                       # max over ranks
    assert all(abs(g[4] - 2 * 100 / 2.5) < 1e-12 for g in got)  # whole-job steps/s
    assert got[0][5] != got[1][5]                              # each rank its own inputs


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.whole_job_rate(1, 10, 2.0) == 5.0
