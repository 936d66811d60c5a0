"""The N>1 path on CPU: two gloo ranks run the replica plumbing the benchmark
uses (barrier, max over ranks, request sharding).  There is no data-path
collective: each rank would own its own pool, tables and caches."""
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


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from paged_kv_cache_39_gb300 import dist as kdist
    r = kdist.init("gloo")
    kdist.barrier()
    # each rank's measured time; the job time is the slowest rank's
    mx = kdist.max_over_ranks(1.5 + rank)
    lo, hi = kdist.shard(10, r)
    kdist.barrier()
    kdist.finalize()
    out.put((rank, r.world_size, mx, lo, hi))


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[1] for x in res] == [2, 2]
    assert [x[2] for x in res] == [2.5, 2.5]
    assert [(x[3], x[4]) for x in res] == [(0, 5), (5, 10)]


@pytest.mark.parametrize("n,world", [(7, 3), (0, 2), (640, 8), (5, 8)])
def test_shard_partitions(n, world):
    from paged_kv_cache_39_gb300.dist import Rank, shard
    spans = [shard(n, Rank(r, r, world)) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == n
    for (a, b), (c, d) in zip(spans, spans[1:]):
        assert b == c and a <= b
    assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1
