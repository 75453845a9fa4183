"""Host-side helpers for running the attention workload on several GPUs.

The (batch, head) problems of attention are independent ("flash_attention.zh"
§8.2: parallelism over batch, heads and query blocks), so N GPUs need no
collective on the data path. Two ways of using them:
  * replicas (weak scaling): every rank runs the whole workload on its own
    seeded data;
  * head shards (strong scaling): the ranks share one seeded batch and each
    runs a contiguous range of its flattened (batch, head) problems
    (``shard``), issued as a few calls over contiguous heads
    (``head_groups``).
The only cross-rank communication is the timing: a barrier before and after
the timed region and a max over ranks of the elapsed time.
"""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class RankInfo:
    rank: int
    world_size: int
    local_rank: int

    @property
    def is_root(self) -> bool:
        return self.rank == 0


def rank_info() -> RankInfo:
    return RankInfo(int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
                    int(os.environ.get("LOCAL_RANK", "0")))


def init(backend: str) -> RankInfo:
    """Joins the process group when launched with more than one rank."""
    info = rank_info()
    if info.world_size > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
    return info


def _dist():
    import torch.distributed as dist
    return dist if dist.is_available() and dist.is_initialized() else None


def barrier() -> None:
    d = _dist()
    if d is not None:
        d.barrier()


def _reduce(x: float, op_name: str, device=None) -> float:
    d = _dist()
    if d is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    d.all_reduce(t, op=getattr(d.ReduceOp, op_name))
    return float(t.item())


def max_over_ranks(x: float, device=None) -> float:
    return _reduce(x, "MAX", device)


def sum_over_ranks(x: float, device=None) -> float:
    return _reduce(x, "SUM", device)


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of rank ``rank``: rank 0 keeps the workload's own seed."""
    return base_seed + 0x1000 * rank


def aggregate_throughput(units_local: float, seconds_local: float, device=None) -> tuple[float, float]:
    """(whole-job units per second, max seconds over ranks): every rank's units
    divided by the slowest rank's time."""
    total_units = sum_over_ranks(units_local, device)
    slowest = max_over_ranks(seconds_local, device)
    return total_units / slowest, slowest


def shard(n_items: int, rank: int, world_size: int) -> range:
    """Contiguous block of ``n_items`` owned by ``rank`` (for strong scaling)."""
    per, extra = divmod(n_items, world_size)
    start = rank * per + min(rank, extra)
    return range(start, start + per + (1 if rank < extra else 0))


def head_groups(items: range, H: int) -> list[tuple[int, int, int, int]]:
    """Split a contiguous range of flattened (batch, head) indices bh = b * H + h
    into calls of the [B, H, N, d] layout: tuples (b0, b1, h0, h1) meaning
    batch entries b0 .. b1-1 with heads h0 .. h1-1, where a tuple spanning
    several batch entries always holds all H heads. Each tuple's slice of a
    contiguous [B, H, N, d] tensor is itself contiguous."""
    lo, hi = items.start, items.stop
    out = []
    while lo < hi:
        b, h = divmod(lo, H)
        if h > 0 or hi - lo < H:  # a partial batch entry
            h1 = min(H, h + (hi - lo))
            out.append((b, b + 1, h, h1))
            lo += h1 - h
        else:  # whole batch entries
            nb = (hi - lo) // H
            out.append((b, b + nb, 0, H))
            lo += nb * H
    return out
