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


def test_head_groups_are_contiguous_calls():
    H = 5
    for n in (1, 4, 5, 6, 14, 15):
        for w in (1, 2, 3, 4):
            for r in range(w):
                items = multi.shard(n, r, w)
                groups = multi.head_groups(items, H)
                got = [b * H + h for (b0, b1, h0, h1) in groups for b in range(b0, b1) for h in range(h0, h1)]
                assert got == list(items)
                for b0, b1, h0, h1 in groups:
                    assert b1 > b0 and h1 > h0
                    assert b1 - b0 == 1 or (h0, h1) == (0, H)  # several batch entries only with every head


def _shard_worker(rank, world, port, result_q):
    """One rank of a head-sharded batch: the oracle forward + backward on its
    own (b, h) problems, taken from its own sub-batch calls the way bench.py
    slices them, gathered on rank 0."""
    import numpy as np
    import oracle
    from exact_io_aware_29_gb300 import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    multi.init("gloo")
    import torch.distributed as dist
    w = synth.small("shard", 3, 5, 40, 8, True, 99, kv_len_range=(10, 40), backward=True)
    lens = w.kv_lens()
    full = [synth.bf16_bits_to_f64(x) for x in (w.q(), w.k(), w.v(), w.do())]
    out = np.full((5, w.B, w.H, w.N, w.d), np.nan)
    owner = np.zeros((w.B, w.H), dtype=np.int64)
    for b0, b1, h0, h1 in multi.head_groups(multi.shard(w.B * w.H, rank, world), w.H):
        q, k, v, do = (x[b0:b1, h0:h1] for x in full)  # the call's sub-batch
        for bb in range(b1 - b0):
            for hh in range(h1 - h0):
                L = int(lens[b0 + bb])
                o, lse = oracle.attention_forward(q[bb, hh], k[bb, hh], v[bb, hh], w.scale, True, L)
                dq, dk, dv = oracle.attention_backward(q[bb, hh], k[bb, hh], v[bb, hh], do[bb, hh], w.scale, True, L)
                out[:, b0 + bb, h0 + hh] = [o, np.repeat(lse[:, None], w.d, 1), dq, dk, dv]
                owner[b0 + bb, h0 + hh] += 1
    got = [None] * world
    dist.all_gather_object(got, (out, owner))
    if rank == 0:
        owners = sum(g[1] for g in got)
        merged = np.where(np.isnan(got[0][0]), got[1][0], got[0][0]) if world == 2 else None
        result_q.put((owners.tolist(), merged))
    dist.destroy_process_group()


def test_gloo_world2_head_shards_reassemble():
    """Two ranks' (b, h) sets are disjoint, cover the batch, and their results
    put together equal the single-rank oracle on every slice."""
    import numpy as np
    import torch.multiprocessing as mp
    import oracle
    from exact_io_aware_29_gb300 import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    owners, merged = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert np.all(np.array(owners) == 1)  # every (b, h) exactly once
    w = synth.small("shard", 3, 5, 40, 8, True, 99, kv_len_range=(10, 40), backward=True)
    lens = w.kv_lens()
    full = [synth.bf16_bits_to_f64(x) for x in (w.q(), w.k(), w.v(), w.do())]
    for b in range(w.B):
        for h in range(w.H):
            L = int(lens[b])
            o, lse = oracle.attention_forward(full[0][b, h], full[1][b, h], full[2][b, h], w.scale, True, L)
            grads = oracle.attention_backward(*(x[b, h] for x in full), w.scale, True, L)
            want = [o, np.repeat(lse[:, None], w.d, 1), *grads]
            for i in range(5):
                assert np.array_equal(merged[i, b, h], want[i])
