"""Multi-rank host logic on CPU (gloo, world size 2): timing aggregation, seeds
and sharding. No GPU and no data-path collective involved."""
import os
import socket

import pytest

from exact_io_aware_29_gb300 import multi


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    info = multi.init("gloo")
    multi.barrier()
    # rank r processed (r + 1) * 10 units in (r + 1) seconds
    rate, slowest = multi.aggregate_throughput(10.0 * (rank + 1), 1.0 * (rank + 1))
    q.put((info.rank, rate, slowest, multi.rank_seed(7, info.rank)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_gloo_world2_aggregation():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # total units 10 + 20 = 30 over the slowest rank's 2 s
    for rank, rate, slowest, seed in out:
        assert rate == pytest.approx(15.0)
        assert slowest == pytest.approx(2.0)
    assert out[0][3] != out[1][3]


def test_single_process_is_identity():
    assert multi.aggregate_throughput(12.0, 3.0) == (4.0, 3.0)
    assert multi.rank_seed(5, 0) == 5


def test_shard_covers_everything_once():
    for n in (1, 7, 64):
        for w in (1, 2, 3, 8):
            got = [i for r in range(w) for i in multi.shard(n, r, w)]
            assert got == list(range(n))
