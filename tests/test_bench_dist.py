"""bench.py's multi-rank host logic on CPU: two gloo ranks, view assignment with no overlap and
the max-over-ranks time / sum-over-ranks entries reduction."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        views = bench.assign_views(rank, world, 10, offset=3)
        t, e = bench.reduce_timing(10.0 + rank, 100 * (rank + 1))
        q.put((rank, views, t, e))
    finally:
        dist.destroy_process_group()


def test_two_ranks_split_views_and_reduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    (r0, v0, t0, e0), (r1, v1, t1, e1) = out
    assert not set(v0) & set(v1) and len(v0) == len(v1) == 10
    assert all(v % 2 == 0 for v in v0) and all(v % 2 == 1 for v in v1)
    assert t0 == t1 == 11.0 and e0 == e1 == 300


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_timing(5.0, 7) == (5.0, 7)
    assert bench.assign_views(0, 1, 3, offset=59) == [59, 0, 1]


def test_launch_count_model():
    import bench
    # 160k Gaussians on 8160 tiles (13 tile bits): projection; clear, depth histogram + 4 passes,
    # slices, expansion, 2 tile passes, ranges, E to the host; tile order, compositing; zeroing,
    # compositing backward, projection backward
    n = bench.launches_per_step(160_000, 1_531_492, 120 * 68)
    assert n == 1 + (1 + 5 + 2 + 2 + 1 + 1) + 2 + 3
