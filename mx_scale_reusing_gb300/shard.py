"""Row sharding across ranks for the MXNorm pass.

Rows (tokens) are independent: each row's codes, scales and inv_rms depend
on that row alone ("MXNorm ...", Resumen tecnico, 2. Metodologia: the
statistics are gathered along the hidden dimension only), so a batch
splits across ranks by contiguous row ranges with no exchange of data.
The only cross-rank traffic is host-side bookkeeping: a barrier and the
maximum of the ranks' step times.
"""
from __future__ import annotations


def row_range(T: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous rows [r0, r1) of rank `rank` when T rows split over `world`
    ranks; the first T % world ranks take one extra row."""
    if world < 1 or not 0 <= rank < world or T < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(T, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def rank_seed(seed: int, rank: int) -> int:
    """Seed of rank `rank`'s own batch when every rank processes a full
    batch of its own (weak scaling)."""
    return seed + 1000 * rank


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank float over the default process group (the
    slowest rank sets a step's time); identity without one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
