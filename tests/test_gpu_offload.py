"""GPU tests of the pinned-host offload pipeline: groups whose residuals and moments live in host
memory step bit-identically to the oracle while their copies overlap other groups' kernels;
slot-ring misuse and injected host-side copy/allocation failures return errors without touching
state and without hanging (failures are made on the host, never on the GPU)."""
import os

import numpy as np
import pytest
import torch

from helpers import OracleNadam
from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(W.NADAM_HP, lr=1e-3)


@pytest.fixture(scope="module")
def eng():
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    return engine


def host_bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16).reshape(-1)


def make_groups(orc, eng, group_shapes, seed, offload):
    oras, grps, tid = [], [], 0
    for shapes in group_shapes:
        masters = [W.master_weights(s, seed, tid + i) for i, s in enumerate(shapes)]
        oras.append(OracleNadam(orc, [m.numpy() for m in masters]))
        grps.append(eng.NadamGroup.from_masters([m.cuda() for m in masters], offload=offload))
        tid += len(shapes)
    return oras, grps


def test_offloaded_groups_bit_exact(orc, eng):
    group_shapes = [[(3000,), (70000,), (20001,)], [(5000,)], [(131075,), (64,)], [(40000,), (1,)]]
    slot = max(eng.offload_slot_bytes([W.numel(s) for s in g]) for g in group_shapes)
    off = eng.OffloadEngine(slot, 3)
    oras, grps = make_groups(orc, eng, group_shapes, 11, off)
    stream = torch.cuda.current_stream()
    for t in range(1, 4):
        grads = []
        tid = 0
        for shapes in group_shapes:
            grads.append([W.grad_bf16(s, 11, tid + i, t, 1e-3, zero_frac=0.01) for i, s in enumerate(shapes)])
            tid += len(shapes)
        grps[0].prefetch()
        for k, (o, g) in enumerate(zip(oras, grps)):
            if k + 1 < len(grps):
                grps[k + 1].prefetch()
            o.step([W.bits16(x).reshape(-1) for x in grads[k]], HP)
            g.step([x.cuda() for x in grads[k]], HP, stream)
    h2d, d2h = off.sync()
    torch.cuda.synchronize()
    assert h2d == d2h > 0
    for o, g in zip(oras, grps):
        for i, ot in enumerate(o.t):
            assert np.array_equal(host_bits(g.weights[i]), ot["hi"])
            assert np.array_equal(host_bits(g.res[i]), ot["lo"])
            if ot["hi"].size > 4096:
                assert np.array_equal(host_bits(g.m[i]), ot["m"])
                assert np.array_equal(host_bits(g.v[i]), ot["v"])
            else:
                assert np.array_equal(g.m[i].numpy(), ot["m"])
                assert np.array_equal(g.v[i].numpy(), ot["v"])
    for g in grps:
        g.close()
    off.close()


def test_slot_ring_and_attach_errors(eng):
    from memory_lean_optimizer_gb300 import lmopt
    off = eng.OffloadEngine(eng.offload_slot_bytes([10000]), 2)
    gs = [eng.NadamGroup.from_masters([torch.zeros(10000, device="cuda")], offload=off) for _ in range(3)]
    gs[0].prefetch()
    gs[1].prefetch()
    with pytest.raises(lmopt.LmoptError) as e:
        gs[2].prefetch()                       # both slots hold groups that have not stepped
    assert e.value.code == lmopt.OPTIM_ESTATE
    g = torch.zeros(10000, dtype=torch.bfloat16, device="cuda")
    gs[0].step([g], HP)
    gs[2].prefetch()                           # slot 0 is free again (device-side ordering)
    gs[1].step([g], HP)
    gs[2].step([g], HP)
    off.sync()
    big = eng.NadamGroup([torch.zeros(20000, dtype=torch.bfloat16, device="cuda")])
    with pytest.raises(lmopt.LmoptError) as e:   # states on the device, not pinned host memory
        lmopt.optim_group_attach_offload(big.handle, off.handle)
    assert e.value.code == lmopt.OPTIM_EINVAL
    with pytest.raises(lmopt.LmoptError) as e:   # engine still has groups attached
        lmopt.optim_offload_destroy(off.handle)
    assert e.value.code == lmopt.OPTIM_ESTATE
    for x in gs + [big]:
        x.close()
    off.close()


def test_injected_failures_leave_state_untouched(eng, monkeypatch):
    from memory_lean_optimizer_gb300 import lmopt
    monkeypatch.setenv("LMOPT_FAULT_INJECT", "alloc")
    with pytest.raises(lmopt.LmoptError) as e:
        eng.OffloadEngine(1 << 20, 2)
    assert e.value.code == lmopt.OPTIM_ENOMEM
    monkeypatch.delenv("LMOPT_FAULT_INJECT")
    off = eng.OffloadEngine(eng.offload_slot_bytes([50000]), 2)
    grp = eng.NadamGroup.from_masters([torch.randn(50000, device="cuda") * 0.02], offload=off)
    g = (torch.randn(50000, device="cuda") * 1e-3).to(torch.bfloat16)
    w0, r0, m0 = grp.weights[0].clone(), grp.res[0].clone(), grp.m[0].clone()
    for what in ("h2d", "d2h"):
        monkeypatch.setenv("LMOPT_FAULT_INJECT", what)
        with pytest.raises(lmopt.LmoptError) as e:
            grp.step([g], HP)
        assert e.value.code == lmopt.OPTIM_ECUDA
        monkeypatch.delenv("LMOPT_FAULT_INJECT")
        off.sync()
        torch.cuda.synchronize()
        assert torch.equal(grp.weights[0], w0) and torch.equal(grp.res[0], r0) and torch.equal(grp.m[0], m0)
        assert lmopt.optim_group_get_step(grp.handle)[0] == 0
    grp.step([g], HP)                          # recovers: the same call now succeeds
    off.sync()
    torch.cuda.synchronize()
    assert not torch.equal(grp.weights[0], w0) or not torch.equal(grp.res[0], r0)
    grp.close()
    off.close()
