"""bench.py's multi-rank plumbing.  The path shards into independent
replicas with no collective on the data path; the bench's only exchange is
the barrier around the timed region and the max of the step time over ranks.
Two gloo ranks on the CPU run those helpers and must agree on the slower
rank's time."""
import multiprocessing as mp
import os
import socket

import pytest


def _rank(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    import torch.distributed as dist

    import bench
    r, ws = bench.dist_init("gloo")
    bench.barrier(ws)
    q.put((r, ws, bench.max_over_ranks(1.5 + rank, ws, device="cpu")))
    bench.barrier(ws)
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slower_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert res == [(0, 2, 2.5), (1, 2, 2.5)]
    assert all(p.exitcode == 0 for p in procs)


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    bench.barrier(1)
    if "WORLD_SIZE" in os.environ and os.environ["WORLD_SIZE"] != "1":
        pytest.skip("run under a launcher")
    assert bench.dist_init("gloo") == (int(os.environ.get("RANK", "0")), 1)
