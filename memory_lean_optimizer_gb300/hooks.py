"""Fused backward pass: step each parameter group from autograd's post-accumulate-grad hooks.

The pages' mechanism: instead of backward-then-step over all gradients, each parameter's
gradient is applied as soon as it is accumulated (``Tensor.register_post_accumulate_grad_hook``),
and optimizer groups step a group of parameters once all of the group's gradients exist, after
which the gradients are dropped ("Fused backward pass" commit, README: "Fused optimizer" and
"Optimizer groups" items).  Here each group is one library group, so one C-ABI call (two kernel
launches) steps every tensor of the group.  Gradient accumulation is not supported, as on the
pages.
"""
from __future__ import annotations

from typing import Callable, Sequence

import torch


def split_groups(params: Sequence[torch.Tensor], n_groups: int) -> list[list[int]]:
    """Contiguous split of the parameter list into n_groups groups of roughly equal element count
    (parameters keep their order, which is roughly the reverse of gradient arrival)."""
    n_groups = max(1, min(n_groups, len(params)))
    total = sum(p.numel() for p in params)
    groups, cur, acc = [], [], 0
    for i, p in enumerate(params):
        cur.append(i)
        acc += p.numel()
        remaining_groups = n_groups - len(groups) - 1
        remaining_params = len(params) - i - 1
        if remaining_groups > 0 and (acc >= total * (len(groups) + 1) / n_groups or remaining_params == remaining_groups):
            groups.append(cur)
            cur = []
    if cur:
        groups.append(cur)
    return groups


class FusedStepper:
    """Registers post-accumulate-grad hooks on `params` and steps each group when its last
    gradient arrives.

    make_group(list_of_params) -> object with .step(grads, hp, stream) (e.g. engine.NadamGroup
    over the parameters' bf16 storage).  After a group steps, its parameters' .grad are set to
    None so that gradient memory is released during the backward pass.
    """

    def __init__(self, params: Sequence[torch.Tensor], n_groups: int, hp: dict,
                 make_group: Callable[[list], object], on_step: Callable | None = None,
                 on_all: Callable | None = None):
        self.params = list(params)
        self.hp = hp
        self.index = split_groups(self.params, n_groups)
        self.groups = [make_group([self.params[i] for i in idx]) for idx in self.index]
        self.group_of = {}
        for gi, idx in enumerate(self.index):
            for i in idx:
                self.group_of[id(self.params[i])] = gi
        self.pending = [len(idx) for idx in self.index]
        self.on_step = on_step
        self.on_all = on_all          # called once every group has stepped (end of a backward)
        self.stepped = 0
        self.steps_taken = [0] * len(self.groups)
        self.ahead = None             # group whose offloaded states were prefetched ahead of its hook
        self.handles = [p.register_post_accumulate_grad_hook(self._hook) for p in self.params]

    def _hook(self, p: torch.Tensor):
        gi = self.group_of[id(p)]
        self.pending[gi] -= 1
        if self.pending[gi] > 0:
            return
        idx = self.index[gi]
        grads = [self.params[i].grad for i in idx]
        if self.on_step is not None:
            self.on_step(gi, grads)
        g = self.groups[gi]
        host = getattr(g, "image", None) is not None   # states in a pinned host image (attach_host)
        if host:
            g.prefetch()                                # nothing if already prefetched
            if self.ahead == gi:
                self.ahead = None
        g.step(grads, self.hp, None)
        if host:
            g.writeback()
            # gradients arrive roughly in reverse parameter order: bring the next group's states
            # in while the backward pass goes on (one group ahead at most, so that with the ring's
            # three slots a group about to step always finds one)
            if self.ahead is None and gi > 0 and getattr(self.groups[gi - 1], "image", None) is not None:
                self.groups[gi - 1].prefetch()
                self.ahead = gi - 1
        self.steps_taken[gi] += 1
        for i in idx:
            self.params[i].grad = None
        self.pending[gi] = len(idx)
        self.stepped += 1
        if self.stepped == len(self.groups):
            self.stepped = 0
            if self.on_all is not None:
                self.on_all()

    def remove(self):
        for h in self.handles:
            h.remove()
        self.handles = []


def attach_fused_nadam(params: Sequence[torch.nn.Parameter], n_groups: int, hp: dict, on_step=None,
                       offload: bool = False) -> FusedStepper:
    """bf16 parameters stepped in place by the fused NAdam+Kahan engine (the parameter's bf16
    storage is the live weight; residuals and u16 moments are allocated per group).  offload:
    each group's residuals and moments live in a pinned host image between its steps (the
    per-group offload calls; each hook prefetches, steps, writes back, and prefetches the group
    whose gradients come next)."""
    from .engine import NadamGroup

    def make(ps):
        g = NadamGroup([p.data for p in ps])
        if offload:
            g.attach_host()
        return g
    return FusedStepper(params, n_groups, hp, make, on_step)


def attach_fused_factored(params: Sequence[torch.nn.Parameter], n_groups: int, hp: dict, on_step=None) -> FusedStepper:
    from .engine import FactoredGroup

    def make(ps):
        return FactoredGroup([p.data for p in ps])
    return FusedStepper(params, n_groups, hp, make, on_step)


def attach_fused_prodigy(params: Sequence[torch.nn.Parameter], n_groups: int, hp: dict, d0: float = 1e-6,
                         slice_p: int = 11, on_step=None) -> FusedStepper:
    """Factored groups in Prodigy mode sharing one step-size estimate d: each group steps from its
    hooks with the current d, and once every group has stepped in a backward pass the
    controller's end of step forms the next d (stepper.prodigy holds the controller).  Every
    parameter must receive a gradient in every backward pass (no frozen parameters): the end of
    step waits for all groups."""
    from .engine import FactoredGroup, ProdigyController
    ctrl = ProdigyController(d0=d0, beta2=hp.get("beta2", 0.999), slice_p=slice_p)

    def make(ps):
        g = FactoredGroup([p.data for p in ps])
        g.attach_prodigy(ctrl)
        return g
    stepper = FusedStepper(params, n_groups, dict(hp, mode=1), make, on_step, on_all=ctrl.end_step)
    stepper.prodigy = ctrl
    return stepper
