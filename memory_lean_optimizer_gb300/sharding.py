"""Data-parallel sharding of the optimizer step across ranks.

The step is element-wise within a tensor and needs nothing from other tensors, so whole groups
can be assigned to ranks with no exchange on the data path: each rank keeps the residuals and
moments of its own groups only (1/N of the optimizer state) and steps them.  If the bf16 weights
are replicated (plain data parallelism), each group's owner broadcasts its updated weights after
the step; if they stay sharded, nothing is exchanged.

A single tensor can also be split into contiguous slices over the ranks (plan_slices,
SlicedNadam).  The u16 codec scale is then the one coupling: it is bounded by maxima over the
whole tensor, so the ranks MAX-reduce three floats per split tensor between the gradient
pre-pass and the update (optim_step_nadam_begin / _end), and the slices step bit-identically to
the unsplit tensor.
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


def my_tensors(sizes: Sequence[int], rank: int, world: int) -> list[int]:
    """Whole tensors (not groups) onto ranks, largest first onto the least-loaded rank: the
    sharding of factored workloads, whose step couples the elements of a tensor (row and column
    means, the RMS clip) but nothing across tensors.  Each rank builds its own groups from its
    tensors; no exchange is needed on the data path.  With many tensors of equal size (the SDXL-like
    workload: 1332 tensors) the ranks end up balanced to within a fraction of a percent, where
    whole groups of 1/10 of the model would not be."""
    return [ti for ti, r in enumerate(assign_groups(sizes, world)) if r == rank]


def replicate_weights(weights_by_group: Sequence[Sequence], owner: Sequence[int], group=None) -> None:
    """After a sharded step: each group's owner broadcasts its updated bf16 weights so that every
    rank holds the same replica (2 bytes per parameter on the wire)."""
    import torch.distributed as dist
    for gi, ws in enumerate(weights_by_group):
        for w in ws:
            # as raw bytes: every backend moves uint8, not every backend moves 16-bit types
            assert w.is_contiguous()
            dist.broadcast(w.view(-1).view(torch.uint8), src=owner[gi], group=group)


SMALL_NUMEL = 4096   # tensors of this many elements or fewer keep fp32 moments


def plan_slices(sizes: Sequence[int], world: int) -> list[list[tuple[int, int, int]]]:
    """Per tensor, its (rank, start, stop) element ranges.  A tensor is split into `world`
    contiguous near-equal slices when every slice keeps more than SMALL_NUMEL elements (so each
    slice keeps the u16 codec, as the whole tensor does); slice starts are multiples of 8 elements
    (16 bytes of bf16), so every slice takes the 128-bit path.  The other tensors go whole,
    largest first, to the least-loaded rank (ties to the lowest rank)."""
    load = [0] * world
    plan: list[list[tuple[int, int, int]]] = [[] for _ in sizes]
    whole = []
    for ti, n in enumerate(sizes):
        if world > 1 and n // world > SMALL_NUMEL + 8:
            bounds = [(n * r // world) // 8 * 8 for r in range(world)] + [n]
            plan[ti] = [(r, bounds[r], bounds[r + 1]) for r in range(world)]
            for r in range(world):
                load[r] += bounds[r + 1] - bounds[r]
        else:
            whole.append(ti)
    for ti in sorted(whole, key=lambda i: (-sizes[i], i)):
        r = min(range(world), key=lambda k: (load[k], k))
        plan[ti] = [(r, 0, sizes[ti])]
        load[r] += sizes[ti]
    return plan


def rank_slices(plan, rank: int) -> tuple[list[tuple[int, int, int]], int]:
    """This rank's (tensor, start, stop) ranges: first one slice of every split tensor, in tensor
    order (the same positions on every rank, so the exchange buffers line up), then the whole
    tensors it owns.  Also returns the number of split tensors."""
    split = [(ti, a, b) for ti, sl in enumerate(plan) if len(sl) > 1 for (r, a, b) in sl if r == rank]
    whole = [(ti, a, b) for ti, sl in enumerate(plan) if len(sl) == 1 for (r, a, b) in sl if r == rank]
    return split + whole, len(split)


class SlicedNadam:
    """NAdam + Kahan + u16 state for this rank's slices of a list of tensors (flat views of the
    full bf16 weights, which every rank holds; residuals and moments exist for the slices only).

    step(): pre-pass, MAX all-reduce of the split tensors' maxima (`all_reduce_max`, a callable
    taking a float32 device tensor, e.g. torch.distributed.all_reduce with ReduceOp.MAX), update.
    Afterwards each slice's owner holds the new weights of its range; gather them with
    share_weights() when the weights are replicated.  With the residual (Kahan) store the result
    is bit-identical to stepping the unsplit tensors; with stochastic rounding each slice draws
    its own random stream (keyed by its position in this rank's group), equally distributed but
    not the same bits."""

    def __init__(self, weights: Sequence[torch.Tensor], residuals: Sequence[torch.Tensor], rank: int, world: int):
        from . import engine
        self.weights = list(weights)
        self.plan = plan_slices([w.numel() for w in self.weights], world)
        self.mine, self.n_split = rank_slices(self.plan, rank)
        self.rank, self.world = rank, world
        ws = [self.weights[ti].view(-1)[a:b] for ti, a, b in self.mine]
        rs = [residuals[ti].view(-1)[a:b] for ti, a, b in self.mine]
        self.group = engine.NadamGroup(ws, rs) if ws else None
        self.exchange = self.group.exchange_buffer() if self.group is not None else None

    def step(self, grads: Sequence[torch.Tensor], hp: dict, all_reduce_max, stream=None):
        if self.group is None:
            if self.n_split:
                raise RuntimeError("a rank without slices cannot take part in the exchange")
            return
        gs = [grads[ti].view(-1)[a:b] for ti, a, b in self.mine]
        self.group.step_begin(gs, hp, self.exchange, stream)
        if self.n_split:
            all_reduce_max(self.exchange[: 3 * self.n_split])
        self.group.step_end(self.exchange, stream)

    def share_weights(self, group=None) -> None:
        """Every rank receives every range's updated bf16 weights from its owner (2 B/param)."""
        import torch.distributed as dist
        for ti, sl in enumerate(self.plan):
            flat = self.weights[ti].view(-1)
            for r, a, b in sl:
                dist.broadcast(flat[a:b].view(torch.uint8), src=r, group=group)
