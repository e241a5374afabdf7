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


@pytest.mark.parametrize("offload", [False, True])
def test_fused_backward_hooks_match_oracle(orc, offload):
    """offload: the groups' residuals and moments live in pinned host images between steps (the
    per-group offload calls from the hooks)."""
    from memory_lean_optimizer_gb300 import build
    from memory_lean_optimizer_gb300.engine import OffloadEngine
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

    stepper = attach_fused_nadam(params, 3, HP, on_step=on_step, offload=offload)
    x = torch.randn(32, 256, device="cuda", dtype=torch.bfloat16)
    for _ in range(3):
        loss = model(x).float().pow(2).mean()
        loss.backward()
    torch.cuda.synchronize()
    if offload:
        OffloadEngine.sync_library_ring()
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


def test_fused_backward_hooks_prodigy_match_oracle(orc):
    """The same in Prodigy mode with d estimated: the controller's end of step runs once every
    group has stepped in a backward pass; d and the weights follow the oracle stepping the captured
    gradients of all groups under one d (d to 1e-5, weights to the factored tolerance)."""
    from memory_lean_optimizer_gb300 import build
    from memory_lean_optimizer_gb300.hooks import attach_fused_prodigy
    build.build()
    torch.manual_seed(1)
    model = torch.nn.Sequential(torch.nn.Linear(256, 512), torch.nn.GELU(), torch.nn.Linear(512, 128)).cuda()
    model = model.to(torch.bfloat16)
    params = list(model.parameters())
    shapes = [tuple(p.shape) for p in params]
    start = [p.detach().float().cpu().numpy().reshape(-1) for p in params]
    captured = {}

    def on_step(gi, grads):
        captured.setdefault(gi, []).append([W.bits16(g).reshape(-1).copy() for g in grads])

    hp = dict(lr=1.0, beta2=0.99, eps1=1e-30, eps2=1e-30, clip_threshold=1.0, weight_decay=0.0, d=1.0)
    stepper = attach_fused_prodigy(params, 2, hp, d0=1e-4, slice_p=3, on_step=on_step)
    x = torch.randn(64, 256, device="cuda", dtype=torch.bfloat16)
    ds = []
    for _ in range(8):
        loss = model(x).float().pow(2).mean()
        loss.backward()
        ds.append(stepper.prodigy.get()[0])
    torch.cuda.synchronize()
    beta3 = stepper.prodigy.beta3
    st = orc.ProdigyState(1e-4, beta3, 3)
    ora = []
    for idx in stepper.index:
        ts = []
        for i in idx:
            hi = (np.frombuffer(start[i].astype(np.float32).tobytes(), np.uint32) >> 16).astype(np.uint16)
            lo = np.zeros_like(hi)
            fac, B, R, C = orc.factored_dims(shapes[i])
            t = dict(hi=hi, lo=lo, shape=shapes[i])
            if fac:
                t["row"], t["col"] = np.zeros(B * R, np.float32), np.zeros(B * C, np.float32)
            else:
                t["V"] = np.zeros(hi.size, np.float32)
            t["p0"], t["s"] = orc.prodigy_snapshot(hi, lo, 3)
            ts.append(t)
        ora.append(ts)
    ds_ref = []
    for k in range(8):
        orc.prodigy_step(st, [(ora[gi], captured[gi][k], dict(hp, mode=1)) for gi in range(len(ora))], k + 1)
        ds_ref.append(st.d.value)
    assert np.allclose(ds, ds_ref, rtol=1e-5, atol=0) and ds_ref[-1] > 1e-4
    lrd = sum(hp["lr"] * float(np.float32(d)) for d in [1e-4] + ds_ref[:-1])
    for gi, idx in enumerate(stepper.index):
        masters = stepper.groups[gi].masters()
        for j, t in enumerate(ora[gi]):
            ref = orc.kahan_merge(t["hi"], t["lo"]).astype(np.float64)
            got = masters[j].cpu().numpy().reshape(-1).astype(np.float64)
            assert np.all(np.abs(got - ref) <= 1e-6 * np.abs(ref) + 2e-5 * lrd), (gi, j)
    stepper.remove()
    stepper.prodigy.close()
