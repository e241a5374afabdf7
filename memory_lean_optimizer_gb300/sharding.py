"""Data-parallel sharding of the optimizer step across ranks.

The step is element-wise within a tensor and needs nothing from other tensors, so whole groups
can be assigned to ranks with no exchange on the data path: each rank keeps the residuals and
moments of its own groups only (1/N of the optimizer state) and steps them.  If the bf16 weights
are replicated (plain data parallelism), each group's owner broadcasts its updated weights after
the step; if they stay sharded, nothing is exchanged.  Splitting one tensor across ranks would
need one MAX all-reduce of three floats per tensor for the codec scale and is not done.
"""
from __future__ import annotations

from typing import Sequence

import torch


def assign_groups(sizes: Sequence[int], world: int) -> list[int]:
    """Owner rank of each group: largest groups first onto the least-loaded rank (ties to the
    lowest rank), so every rank ends with nearly the same number of parameters."""
    load = [0] * world
    owner = [0] * len(sizes)
    for gi in sorted(range(len(sizes)), key=lambda i: (-sizes[i], i)):
        r = min(range(world), key=lambda k: (load[k], k))
        owner[gi] = r
        load[r] += sizes[gi]
    return owner


def my_groups(sizes: Sequence[int], rank: int, world: int) -> list[int]:
    return [gi for gi, r in enumerate(assign_groups(sizes, world)) if r == rank]


def replicate_weights(weights_by_group: Sequence[Sequence], owner: Sequence[int], group=None) -> None:
    """After a sharded step: each group's owner broadcasts its updated bf16 weights so that every
    rank holds the same replica (2 bytes per parameter on the wire)."""
    import torch.distributed as dist
    for gi, ws in enumerate(weights_by_group):
        for w in ws:
            # as raw bytes: every backend moves uint8, not every backend moves 16-bit types
            assert w.is_contiguous()
            dist.broadcast(w.view(-1).view(torch.uint8), src=owner[gi], group=group)
