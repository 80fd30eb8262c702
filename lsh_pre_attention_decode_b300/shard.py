"""Placement of independent HashEvict units on ranks (one process per GPU).

Every (layer, batch, KV head) unit owns its cache, codes, eviction decision and
attention (HashEvict paper, technical framework: the steps are per head and per
sequence), so a multi-GPU run only partitions units: no data crosses ranks and
no collective sits on the data path.  The only collective is the host-side
max-over-ranks of a timing, taken after the timed region.
"""
from __future__ import annotations


def layer_shard(rank: int, world: int, layers_per_rank: int) -> list[int]:
    """Layers owned by `rank`: rank r takes r*L .. r*L+L-1 (weak scaling: every
    rank holds the same amount of work whatever the world size)."""
    if world < 1 or not 0 <= rank < world or layers_per_rank < 1:
        raise ValueError(f"bad shard request rank={rank} world={world} L={layers_per_rank}")
    return [rank * layers_per_rank + i for i in range(layers_per_rank)]


def batch_shard(rank: int, world: int, batch: int) -> range:
    """Contiguous batch rows owned by `rank` when one layer's batch is split
    (strong scaling); the first batch % world ranks take one extra row."""
    if world < 1 or not 0 <= rank < world or batch < 0:
        raise ValueError(f"bad shard request rank={rank} world={world} batch={batch}")
    base, extra = divmod(batch, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a host float over the ranks of the default process group (the
    value itself when no group is initialised).  `device` is where the reduced
    tensor lives: a CUDA device for NCCL, None (CPU) for gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
