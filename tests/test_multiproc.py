"""bench.py's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

The library shards only as independent replicas (every (sequence, head)
unit and every prefill sequence is independent, so there is no exchange
step); across ranks the bench only synchronises (barrier) and reduces its
timings (maximum over ranks).  No GPU needed."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(1.5 + rank, world)       # each rank's own "elapsed time"
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)
