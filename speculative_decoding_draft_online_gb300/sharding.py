"""Splitting a verification batch across ranks.

Sequences are independent, so B sequences shard with no exchange inside the
verification itself: rank r takes sequences [B*r/W, B*(r+1)/W) and passes the
index of its first sequence as `sequence_offset`, which makes its random draws
those of the whole batch.  Only the small [B]-sized outputs are gathered.
"""
from __future__ import annotations

from typing import Tuple

import torch


def shard_bounds(B: int, rank: int, world: int) -> Tuple[int, int]:
    """[start, stop) of the sequences rank `rank` of `world` verifies."""
    if not (0 <= rank < world) or B < 0:
        raise ValueError(f"bad shard request B={B} rank={rank} world={world}")
    return B * rank // world, B * (rank + 1) // world


def gather_rows(local: torch.Tensor, B: int, world: int, group=None) -> torch.Tensor:
    """All-gather per-sequence rows (shape [b_r, ...]) of every rank into [B, ...].

    Shards may differ in size by one; they are padded to the largest before the
    collective and trimmed after.
    """
    import torch.distributed as dist
    rows = max(shard_bounds(B, r, world)[1] - shard_bounds(B, r, world)[0] for r in range(world))
    pad = torch.full((rows,) + tuple(local.shape[1:]), -1, dtype=local.dtype, device=local.device)
    pad[: local.shape[0]] = local
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    out = []
    for r in range(world):
        a, b = shard_bounds(B, r, world)
        out.append(parts[r][: b - a])
    return torch.cat(out, dim=0)
