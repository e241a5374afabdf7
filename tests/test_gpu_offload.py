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


# ---------------------------------------------------------------- every offloadable group kind
ADAN_HP = dict(lr=3.3e-5, beta1=0.02, beta2=0.08, beta3=0.01, eps=1e-8, weight_decay=0.02)
KINDS = ["nadam-u16", "nadam-f24", "adan-fp32", "adan-f24"]


def _bytes(a):
    if isinstance(a, torch.Tensor):
        return a.contiguous().cpu().view(torch.uint8).numpy().reshape(-1)
    return np.ascontiguousarray(a).view(np.uint8).reshape(-1)


class OracleGroup:
    """Oracle states of one group of any offloadable kind, stepped tensor by tensor."""

    def __init__(self, orc, masters, kind):
        self.orc, self.kind, self.t = orc, kind, []
        self.nstate = orc.NadamState(len(masters))
        self.mp, self.steps = 1.0, 0
        for x in masters:
            hi, lo = orc.kahan_split(np.ascontiguousarray(x, np.float32).reshape(-1))
            n = hi.size
            d = dict(hi=hi, lo=lo)
            if kind == "nadam-u16":
                d["m"] = np.zeros(n, np.float32) if n <= 4096 else np.full(n, 32768, np.uint16)
                d["v"] = np.zeros(n, np.float32) if n <= 4096 else np.zeros(n, np.uint16)
            elif kind == "nadam-f24":
                d["m"] = np.zeros(n, np.float32) if n <= 4096 else np.zeros(orc.f24_nbytes(n), np.uint8)
                d["v"] = np.zeros(n, np.float32) if n <= 4096 else np.zeros(orc.f24_nbytes(n), np.uint8)
            else:
                d["m"] = (np.zeros(orc.adan_f24_nbytes(n), np.uint8) if kind == "adan-f24"
                          else np.zeros(3 * orc.adan_plane(n), np.float32))
                d["v"] = np.zeros(n, np.uint16)
            self.t.append(d)

    def step(self, grads):
        self.steps += 1
        orc, t = self.orc, self.steps
        g = [W.bits16(x).reshape(-1) for x in grads]
        if self.kind == "nadam-u16":
            orc.nadam_group_step(self.t, g, self.nstate, t, HP)
        elif self.kind == "nadam-f24":
            k, self.mp = orc.nadam_scalars(t, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"],
                                           HP["wd_mode"] == 1, HP["nesterov"], HP["momentum_decay"], self.mp)
            for d, gg in zip(self.t, g):
                orc.nadam_step_tensor_f24(d["hi"], d["lo"], d["m"], d["v"], gg, k)
        else:
            k = orc.adan_scalars(ADAN_HP["lr"], ADAN_HP["beta1"], ADAN_HP["beta2"], ADAN_HP["beta3"],
                                 ADAN_HP["eps"], ADAN_HP["weight_decay"])
            fn = orc.adan_step_tensor_f24 if self.kind == "adan-f24" else orc.adan_step_tensor
            for d, gg in zip(self.t, g):
                fn(d["hi"], d["lo"], d["m"], d["v"], gg, t, k)


def make_group(eng, masters, kind, offload=None):
    fam, states = kind.split("-")
    if fam == "nadam":
        return eng.NadamGroup.from_masters(masters, offload=offload, states=states)
    return eng.AdanGroup.from_masters(masters, states=states, offload=offload)


def step_group(grp, kind, grads, stream):
    grp.step(grads, HP if kind.startswith("nadam") else ADAN_HP, stream)


def assert_group_equal(o, grp, tag):
    states = (grp.res, grp.m, grp.v) if o.kind.startswith("nadam") else (grp.res, grp.mvn, grp.gprev)
    for i, d in enumerate(o.t):
        assert np.array_equal(host_bits(grp.weights[i]), d["hi"]), f"{tag}: tensor {i} weights"
        for name, got, want in zip(("residual", "m", "v"), states, (d["lo"], d["m"], d["v"])):
            assert np.array_equal(_bytes(got[i]), _bytes(want)), f"{tag}: tensor {i} {name}"


GROUP_SHAPES = [[(3000,), (70000,), (20001,)], [(5000,), (0,)], [(131075,), (64,)], [(40000,), (1,)]]


def _grads(group_shapes, seed, t):
    out, tid = [], 0
    for shapes in group_shapes:
        out.append([W.grad_bf16(s, seed, tid + i, t, 1e-3, zero_frac=0.01) for i, s in enumerate(shapes)])
        tid += len(shapes)
    return out


@pytest.mark.parametrize("kind", KINDS)
def test_engine_offload_every_kind(orc, eng, kind):
    """Groups of every offloadable kind attached to an engine (states in pinned host buffers, the
    step prefetching and writing back): bit-identical to the oracle after 3 steps."""
    from memory_lean_optimizer_gb300 import lmopt
    kid = {"nadam-u16": lmopt.OPTIM_KIND_NADAM, "nadam-f24": lmopt.OPTIM_KIND_NADAM_F24,
           "adan-fp32": lmopt.OPTIM_KIND_ADAN, "adan-f24": lmopt.OPTIM_KIND_ADAN_F24}[kind]
    seed = 31
    off = eng.OffloadEngine(max(eng.offload_slot_bytes([W.numel(s) for s in g], kind=kid) for g in GROUP_SHAPES), 3)
    oras, grps, tid = [], [], 0
    for shapes in GROUP_SHAPES:
        masters = [W.master_weights(s, seed, tid + i) for i, s in enumerate(shapes)]
        oras.append(OracleGroup(orc, [m.numpy() for m in masters], kind))
        grps.append(make_group(eng, [m.cuda() for m in masters], kind, offload=off))
        tid += len(shapes)
    stream = torch.cuda.current_stream()
    for t in range(1, 4):
        grads = _grads(GROUP_SHAPES, seed, t)
        grps[0].prefetch()
        for k, (o, g) in enumerate(zip(oras, grps)):
            if k + 1 < len(grps):
                grps[k + 1].prefetch()
            o.step(grads[k])
            step_group(g, kind, [x.cuda() for x in grads[k]], stream)
    off.sync()
    torch.cuda.synchronize()
    for k, (o, g) in enumerate(zip(oras, grps)):
        assert_group_equal(o, g, f"{kind} group {k}")
    for g in grps:
        g.close()
    off.close()


@pytest.mark.parametrize("kind", KINDS)
def test_attach_host_pipeline_every_kind(orc, eng, kind):
    """The per-group offload calls: each group's states moved into one pinned host image
    (optim_group_attach_host); per step prefetch(k+1) on a copy-in stream before step(k), and
    write-back(k) on a copy-out stream after it, through the library's own staging ring.  The
    images equal the oracle's states bit for bit after 3 steps, and the device buffers named at
    create are no longer used (they are dropped by attach_host)."""
    seed = 32
    oras, grps, tid = [], [], 0
    for shapes in GROUP_SHAPES:
        masters = [W.master_weights(s, seed, tid + i) for i, s in enumerate(shapes)]
        oras.append(OracleGroup(orc, [m.numpy() for m in masters], kind))
        g = make_group(eng, [m.cuda() for m in masters], kind)
        g.attach_host()
        grps.append(g)
        tid += len(shapes)
    stream = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    for t in range(1, 4):
        grads = _grads(GROUP_SHAPES, seed, t)
        grps[0].prefetch(cin)
        for k, (o, g) in enumerate(zip(oras, grps)):
            if k + 1 < len(grps):
                grps[k + 1].prefetch(cin)
            o.step(grads[k])
            step_group(g, kind, [x.cuda() for x in grads[k]], stream)
            g.writeback(cout)
    torch.cuda.synchronize()
    for k, (o, g) in enumerate(zip(oras, grps)):
        assert_group_equal(o, g, f"{kind} group {k}")
    for g in grps:
        g.close()


def test_attach_host_errors_and_ring_growth(orc, eng):
    """Misuse of the per-group offload calls returns an error and changes nothing: an image too
    small or not pinned, a factored group, a step before prefetch, a write-back without a slot,
    growing the library's ring while a group's states are on the device.  A larger group then
    grows the ring, and both groups step bit-identically to the oracle."""
    from memory_lean_optimizer_gb300 import lmopt
    small = eng.NadamGroup.from_masters([W.master_weights((6000,), 33, 0).cuda()])
    total, offs = lmopt.optim_offload_layout(small.handle, 1)
    assert total == 3 * 12032 and offs == [(0, 12032, 24064)]     # 12000 bytes each, 256-byte aligned
    pinned = torch.zeros(total, dtype=torch.uint8, pin_memory=True)
    dev = torch.zeros(total, dtype=torch.uint8, device="cuda")
    for ptr, nb in ((pinned.data_ptr(), total - 1), (dev.data_ptr(), total)):
        with pytest.raises(lmopt.LmoptError) as e:
            lmopt.optim_group_attach_host(small.handle, ptr, nb)
        assert e.value.code == lmopt.OPTIM_EINVAL
    fac = eng.FactoredGroup.from_masters([torch.zeros(64, 64, device="cuda")])
    with pytest.raises(lmopt.LmoptError) as e:
        lmopt.optim_offload_layout(fac.handle, 1)
    assert e.value.code == lmopt.OPTIM_EINVAL
    fac.close()
    with pytest.raises(lmopt.LmoptError) as e:         # not attached
        small.writeback()
    assert e.value.code == lmopt.OPTIM_EINVAL
    ora_s = OracleGroup(orc, [W.master_weights((6000,), 33, 0).numpy()], "nadam-u16")
    small.attach_host()
    g1 = W.grad_bf16((6000,), 33, 0, 1, 1e-3)
    with pytest.raises(lmopt.LmoptError) as e:         # no prefetch yet
        small.step([g1.cuda()], HP)
    assert e.value.code == lmopt.OPTIM_ESTATE
    with pytest.raises(lmopt.LmoptError) as e:         # holds no slot
        small.writeback()
    assert e.value.code == lmopt.OPTIM_ESTATE
    assert lmopt.optim_group_get_step(small.handle)[0] == 0
    small.prefetch()
    big = eng.NadamGroup.from_masters([W.master_weights((50000,), 33, 1).cuda()])
    with pytest.raises(lmopt.LmoptError) as e:         # the ring must grow, a slot is held
        big.attach_host()
    assert e.value.code == lmopt.OPTIM_ESTATE
    small.step([g1.cuda()], HP)
    ora_s.step([g1])
    small.writeback()
    ora_b = OracleGroup(orc, [W.master_weights((50000,), 33, 1).numpy()], "nadam-u16")
    big.attach_host()                                  # grows the ring (no slot held now)
    for t in (2, 3):
        gs = W.grad_bf16((6000,), 33, 0, t, 1e-3)
        gb = W.grad_bf16((50000,), 33, 1, t, 1e-3)
        small.prefetch()
        big.prefetch()
        small.step([gs.cuda()], HP)
        big.step([gb.cuda()], dict(HP))
        small.writeback()
        big.writeback()
        ora_s.step([gs])
        ora_b.step([gb])
    eng.OffloadEngine.sync_library_ring()
    torch.cuda.synchronize()
    assert_group_equal(ora_s, small, "small group")
    # the big group stepped twice (t = 1, 2 of its own counter)
    assert_group_equal(ora_b, big, "big group")
    small.close()
    big.close()
