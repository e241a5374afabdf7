"""Fused backward pass on the GPU: a small bf16 model whose parameters are stepped by the engine
from autograd's post-accumulate-grad hooks, one library call per group, as soon as the group's
last gradient exists.  The gradients each group receives are captured and replayed through the
oracle: weights, residuals and moment codes must match bit for bit."""
import numpy as np
import pytest
import torch

from helpers import OracleNadam, assert_nadam_equal
from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(W.NADAM_HP, lr=1e-3)


def test_fused_backward_hooks_match_oracle(orc):
    from memory_lean_optimizer_gb300 import build
    from memory_lean_optimizer_gb300.hooks import attach_fused_nadam
    build.build()
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(256, 512), torch.nn.GELU(), torch.nn.Linear(512, 128),
                                torch.nn.GELU(), torch.nn.Linear(128, 64)).cuda().to(torch.bfloat16)
    params = list(model.parameters())
    start = [p.detach().float().cpu().numpy().reshape(-1) for p in params]
    captured = {}

    def on_step(gi, grads):
        captured.setdefault(gi, []).append([W.bits16(g).reshape(-1).copy() for g in grads])

    stepper = attach_fused_nadam(params, 3, HP, on_step=on_step)
    x = torch.randn(32, 256, device="cuda", dtype=torch.bfloat16)
    for _ in range(3):
        loss = model(x).float().pow(2).mean()
        loss.backward()
    torch.cuda.synchronize()
    assert all(p.grad is None for p in params)
    assert all(len(captured[gi]) == 3 for gi in range(len(stepper.groups)))
    for gi, idx in enumerate(stepper.index):
        # the live weight starts as the bf16 parameter, residual zero (exactly what the group holds)
        ora = OracleNadam(orc, [start[i] for i in idx])
        for t in ora.t:
            t["lo"][:] = 0
        for grads in captured[gi]:
            ora.step(grads, HP)
        assert_nadam_equal(ora, stepper.groups[gi], f"group {gi}")
        for i, p in zip(idx, [params[i] for i in idx]):
            assert p.data.data_ptr() == stepper.groups[gi].weights[idx.index(i)].data_ptr()
    stepper.remove()
