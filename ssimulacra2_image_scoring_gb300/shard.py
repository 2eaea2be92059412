"""Frame sharding across ranks (one process per GPU).

Frames are independent and each yields 8 bytes, so a frame sequence splits
into contiguous ranges, one per rank, with no exchange on the data path;
only the scores are gathered, on the host, at the end.
"""
from __future__ import annotations

import numpy as np


def frame_range(n_frames: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of this rank's frames: contiguous, sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or n_frames < 0:
        raise ValueError(f"bad split: {n_frames} frames, world {world}, rank {rank}")
    base, extra = divmod(n_frames, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def score_sharded(score_fn, ref, dis, group=None) -> np.ndarray:
    """Scores this rank's frame range with ``score_fn(ref_part, dis_part)``
    (any callable returning one float64 per frame, e.g. ``Scorer.score``) and
    returns every rank's scores in frame order, gathered through
    torch.distributed on the host."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    a, b = frame_range(len(ref), world, rank)
    mine = np.asarray(score_fn(ref[a:b], dis[a:b]), dtype=np.float64)
    parts: list = [None] * world
    dist.all_gather_object(parts, (a, mine), group=group)
    out = np.empty(len(ref), np.float64)
    for start, sc in parts:
        out[start:start + len(sc)] = sc
    return out
