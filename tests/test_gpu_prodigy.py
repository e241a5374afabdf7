"""GPU parity of Prodigy's step-size estimate d over FACTORED groups (mode 1) against the oracle,
through the C ABI: two groups sharing one controller, mixed tensor classes (wide matrices, batched
matrices, 3x3 convolutions, vectors), sliced and unsliced statistics.

Tolerances, derived from the arithmetic:
  s (sampled denominators) : the same fp32 operations per element, with fl(lr d_k^2) from d_k:
                             1e-5 of the tensor's largest |s| (see the check)
  d                        : 1e-5 relative.  Both sides sum the same fp32 terms; the oracle in
                             double in element order, the kernels in fp32 over 32 terms per thread
                             and double beyond (a few fp32 roundings of the partial sums), and the
                             weights they were computed from carry the factored step's own
                             ~1e-6 differences.
  fp32 masters             : |w - w_ref| <= 1e-6 |w_ref| + 2e-5 * sum_k lr d_k  (the update is
                             lr d_k per step; a 1e-5-relative difference in d_k, plus the factored
                             step's 1e-6)
"""
import numpy as np
import pytest
import torch

from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(beta2=0.99, decay_rate=-0.8, eps1=1e-30, eps2=1e-30, d=1.0, clip_threshold=1.0, weight_decay=0.0,
          mode=1)
GROUPS = [[(64, 80), (3, 40, 72), (8, 8, 3, 3), (300,), (45, 50, 3, 3)],
          [(1000, 640), (600, 2, 2), (77,), (5000,)]]


@pytest.fixture(scope="module")
def eng():
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    return engine


def oracle_tensor(orc, x, shape, slice_p):
    x = np.ascontiguousarray(x, np.float32).reshape(-1)
    hi, lo = orc.kahan_split(x)
    fac, B, R, C = orc.factored_dims(shape)
    t = dict(hi=hi, lo=lo, shape=shape)
    if fac:
        t["row"] = np.zeros(B * R, np.float32)
        t["col"] = np.zeros(B * C, np.float32)
    else:
        t["V"] = np.zeros(x.size, np.float32)
    t["p0"], t["s"] = orc.prodigy_snapshot(hi, lo, slice_p)
    return t


def run(orc, eng, slice_p, steps, hps, d0=1e-4, seed=70):
    beta3 = float(np.float32(np.sqrt(0.99)))
    st = orc.ProdigyState(d0, beta3, slice_p)
    ctrl = eng.ProdigyController(d0=d0, beta3=beta3, slice_p=slice_p)
    ora, grps, bias = [], [], []
    tid = 0
    for shapes in GROUPS:
        masters = [W.master_weights(s, seed, tid + i) for i, s in enumerate(shapes)]
        ora.append([oracle_tensor(orc, m.numpy(), s, slice_p) for m, s in zip(masters, shapes)])
        grp = eng.FactoredGroup.from_masters([m.cuda() for m in masters])
        grp.attach_prodigy(ctrl)
        grps.append(grp)
        bias.append([W.grad_bf16(s, seed + 1, tid + i, 0, 1e-3).float() for i, s in enumerate(shapes)])
        tid += len(shapes)
    ds, ds_ref, lrd = [], [], 0.0
    for t in range(1, steps + 1):
        step_groups = []
        tid = 0
        for gi, shapes in enumerate(GROUPS):
            # a persistent component makes the displacement correlate with the gradients, so d grows
            grads = [(bias[gi][i] + W.grad_bf16(s, seed, tid + i, t, 3e-4).float()).to(torch.bfloat16)
                     for i, s in enumerate(shapes)]
            tid += len(shapes)
            step_groups.append(([W.bits16(g).reshape(-1) for g in grads], grads))
        lrd += max(h["lr"] for h in hps) * st.d32
        orc.prodigy_step(st, [(ora[gi], step_groups[gi][0], hps[gi]) for gi in range(len(GROUPS))], t)
        for gi, grp in enumerate(grps):
            grp.step([g.cuda() for g in step_groups[gi][1]], hps[gi])
        ctrl.end_step()
        ds.append(ctrl.get()[0])
        ds_ref.append(st.d.value)
    torch.cuda.synchronize()
    return ora, grps, ctrl, ds, ds_ref, lrd


def check(orc, ora, grps, ds, ds_ref, lrd):
    assert np.allclose(ds, ds_ref, rtol=1e-5, atol=0), (ds, ds_ref)
    from memory_lean_optimizer_gb300 import lmopt
    for og, grp in zip(ora, grps):
        masters = grp.masters()
        for i, ot in enumerate(og):
            ref = orc.kahan_merge(ot["hi"], ot["lo"]).astype(np.float64)
            got = masters[i].cpu().numpy().reshape(-1).astype(np.float64)
            tol = 1e-6 * np.abs(ref) + 2e-5 * lrd
            bad = np.abs(got - ref) > tol
            assert not bad.any(), f"{ot['shape']}: {bad.sum()} masters out of tolerance"
            assert np.array_equal(grp.p0[i][:ot["p0"].size].cpu().numpy().view(np.uint32), ot["p0"].view(np.uint32))
            # s = sum_j beta3^(k-j) fl(lr d_j^2) g_j: a 1e-5-relative difference in d_j moves it by
            # up to 1e-5 of the sum of the terms' magnitudes, which cancellation can leave far
            # above |s| itself; bounded here by the tensor's largest |s|
            s_got = grp.s[i][:ot["s"].size].cpu().numpy().astype(np.float64)
            s_ref = ot["s"].astype(np.float64)
            err = np.abs(s_got - s_ref)
            assert np.all(err <= 1e-5 * np.abs(s_ref) + 1e-5 * np.abs(s_ref).max()), \
                f"{ot['shape']}: s differs (max error {err.max():.3e}, max |s| {np.abs(s_ref).max():.3e})"
        assert lmopt.optim_query_nonfinite(grp.handle) == 0


@pytest.mark.parametrize("slice_p", [1, 3, 11])
def test_prodigy_d_adaptation_parity(orc, eng, slice_p):
    hps = [dict(HP, lr=1.0), dict(HP, lr=0.5, weight_decay=0.01)]
    ora, grps, ctrl, ds, ds_ref, lrd = run(orc, eng, slice_p, 8, hps)
    assert ds_ref[0] == 1e-4 and ds_ref[-1] > 2e-4          # d grows within the run
    check(orc, ora, grps, ds, ds_ref, lrd)
    ctrl.close()


def _pd_grads(shapes, gi, tid0, t, seed):
    bias = [W.grad_bf16(s, seed + 1, tid0 + i, 0, 1e-3).float() for i, s in enumerate(shapes)]
    return [(bias[i] + W.grad_bf16(s, seed, tid0 + i, t, 3e-4).float()).to(torch.bfloat16).cuda()
            for i, s in enumerate(shapes)]


def _pd_build(eng, slice_p, d0, beta3, seed):
    ctrl = eng.ProdigyController(d0=d0, beta3=beta3, slice_p=slice_p)
    grps, tid = [], 0
    for shapes in GROUPS:
        masters = [W.master_weights(s, seed, tid + i) for i, s in enumerate(shapes)]
        grp = eng.FactoredGroup.from_masters([m.cuda() for m in masters])
        grp.attach_prodigy(ctrl)
        grps.append(grp)
        tid += len(shapes)
    return ctrl, grps


def _pd_steps(ctrl, grps, hps, t0, t1, seed):
    for t in range(t0, t1 + 1):
        tid = 0
        for gi, (shapes, grp) in enumerate(zip(GROUPS, grps)):
            grp.step(_pd_grads(shapes, gi, tid, t, seed), hps[gi])
            tid += len(shapes)
        ctrl.end_step()


def test_prodigy_checkpoint_resume_bit_identical(orc, eng):
    """k steps, save (weights, residuals, R and C or V, p0, s, d, r, step), restore into new groups
    and a new controller attached without a snapshot: N-k more steps equal N uninterrupted steps
    bit for bit (every reduction on this path has a fixed order)."""
    from memory_lean_optimizer_gb300 import lmopt
    slice_p, d0, seed, N, k = 3, 1e-4, 72, 8, 4
    hps = [dict(HP, lr=1.0), dict(HP, lr=0.5, weight_decay=0.01)]
    beta3 = float(np.float32(np.sqrt(0.99)))
    ctrl, grps = _pd_build(eng, slice_p, d0, beta3, seed)
    _pd_steps(ctrl, grps, hps, 1, N, seed)
    ref = [[(w.clone(), r.clone()) for w, r in zip(g.weights, g.res)] for g in grps]
    d_ref = ctrl.get()
    ctrl.close()

    ctrl, grps = _pd_build(eng, slice_p, d0, beta3, seed)
    _pd_steps(ctrl, grps, hps, 1, k, seed)
    saved = [dict(w=[w.clone() for w in g.weights], res=[r.clone() for r in g.res],
                  row=[x.clone() if x is not None else None for x in g.row], col=[x.clone() for x in g.col],
                  p0=[x.clone() for x in g.p0], s=[x.clone() for x in g.s]) for g in grps]
    d, r = ctrl.get()
    ctrl.close()

    ctrl = eng.ProdigyController(d0=d0, beta3=beta3, slice_p=slice_p)
    ctrl.set(d, r)
    grps = []
    for sv in saved:
        grp = eng.FactoredGroup(sv["w"], sv["res"])
        for dst, src in zip(grp.row + grp.col, sv["row"] + sv["col"]):
            if dst is not None:
                dst.copy_(src)
        lmopt.optim_group_set_step(grp.handle, k, 1.0)
        grp.step_count = k
        grp.attach_prodigy(ctrl, p0=sv["p0"], s=sv["s"])
        grps.append(grp)
    _pd_steps(ctrl, grps, hps, k + 1, N, seed)
    assert ctrl.get() == d_ref
    for g, rg in zip(grps, ref):
        for w, r, (w0, r0) in zip(g.weights, g.res, rg):
            assert torch.equal(w, w0) and torch.equal(r, r0)
    ctrl.close()


def test_prodigy_api_errors(eng):
    from memory_lean_optimizer_gb300 import lmopt
    with pytest.raises(lmopt.LmoptError):
        lmopt.optim_prodigy_create(0.0, 0.9, 1)
    with pytest.raises(lmopt.LmoptError):
        lmopt.optim_prodigy_create(1e-6, 1.0, 1)
    with pytest.raises(lmopt.LmoptError):
        lmopt.optim_prodigy_create(1e-6, 0.9, 0)
    assert lmopt.optim_prodigy_slice_len(400, 3) == 192 and lmopt.optim_prodigy_slice_len(-1, 3) == -1
    ctrl = eng.ProdigyController(d0=1e-6, slice_p=4)
    grp = eng.FactoredGroup.from_masters([torch.randn(64, 32, device="cuda") * 0.02])
    grp.attach_prodigy(ctrl)
    with pytest.raises(lmopt.LmoptError) as e:          # destroy while a group is attached
        lmopt.optim_prodigy_destroy(ctrl.handle)
    assert e.value.code == lmopt.OPTIM_ESTATE
    g = [torch.zeros(64, 32, dtype=torch.bfloat16, device="cuda")]
    with pytest.raises(lmopt.LmoptError):                # attached groups step in mode 1
        grp.step(g, dict(HP, lr=1.0, mode=0))
    with pytest.raises(lmopt.LmoptError) as e:           # attaches once
        grp.attach_prodigy(ctrl)
    assert e.value.code == lmopt.OPTIM_ESTATE
    grp.step(g, dict(HP, lr=1.0))
    ctrl.end_step()
    assert ctrl.get()[0] == 1e-6                          # zero gradients: s stays 0, d unchanged
    ctrl.close()


def test_two_ranks_share_d_through_reduce_finish(orc, eng):
    """Two controllers (as two data-parallel ranks on one GPU, stepped one after the other), one
    group each: their reduce() sums are added and passed to both finish() calls, so both hold the
    same d, which follows the oracle stepping both groups under one d."""
    from memory_lean_optimizer_gb300 import lmopt
    slice_p, d0, seed = 3, 1e-4, 71
    hps = [dict(HP, lr=1.0), dict(HP, lr=0.5)]
    beta3 = float(np.float32(np.sqrt(0.99)))
    st = orc.ProdigyState(d0, beta3, slice_p)
    ctrls = [eng.ProdigyController(d0=d0, beta3=beta3, slice_p=slice_p) for _ in GROUPS]
    ora, grps, bias = [], [], []
    tid = 0
    for gi, shapes in enumerate(GROUPS):
        masters = [W.master_weights(s, seed, tid + i) for i, s in enumerate(shapes)]
        ora.append([oracle_tensor(orc, m.numpy(), s, slice_p) for m, s in zip(masters, shapes)])
        grp = eng.FactoredGroup.from_masters([m.cuda() for m in masters])
        grp.attach_prodigy(ctrls[gi])
        grps.append(grp)
        bias.append([W.grad_bf16(s, seed + 1, tid + i, 0, 1e-3).float() for i, s in enumerate(shapes)])
        tid += len(shapes)
    for t in range(1, 9):
        step_groups = []
        tid = 0
        for gi, shapes in enumerate(GROUPS):
            grads = [(bias[gi][i] + W.grad_bf16(s, seed, tid + i, t, 3e-4).float()).to(torch.bfloat16)
                     for i, s in enumerate(shapes)]
            tid += len(shapes)
            step_groups.append(grads)
        orc.prodigy_step(st, [(ora[gi], [W.bits16(g).reshape(-1) for g in step_groups[gi]], hps[gi])
                              for gi in range(len(GROUPS))], t)
        parts = []
        for gi, grp in enumerate(grps):
            grp.step([g.cuda() for g in step_groups[gi]], hps[gi])
            buf = torch.empty(2, dtype=torch.float64, device="cuda")
            lmopt.optim_prodigy_reduce(ctrls[gi].handle, buf.data_ptr(), 0)
            parts.append(buf)
        total = parts[0] + parts[1]
        for c in ctrls:
            lmopt.optim_prodigy_finish(c.handle, total.data_ptr(), 0)
        da, db = ctrls[0].get()[0], ctrls[1].get()[0]
        assert da == db
        assert abs(da - st.d.value) <= 1e-5 * st.d.value, (t, da, st.d.value)
    assert st.d.value > 2 * d0
    for c in ctrls:
        c.close()


def test_prodigy_misaligned_buffers_and_empty_tensors(orc, eng):
    """Weights, residuals and gradients 2 bytes aligned and p0 / s 4 bytes (not 16) aligned take
    the statistics kernel's element-by-element path; empty tensors add nothing.  d, s and the
    weights follow the oracle as in the aligned case."""
    from helpers import alloc_offset, cuda_bits
    from memory_lean_optimizer_gb300 import lmopt
    shapes = [(96, 64), (40, 50, 3, 3), (700,), (0, 64), (0,), (33, 40)]
    seed, steps, slice_p, d0 = 9, 6, 3, 1e-4
    hp = dict(HP, lr=1.0)
    beta3 = float(np.float32(np.sqrt(0.99)))
    st = orc.ProdigyState(d0, beta3, slice_p)
    masters = [W.master_weights(s, seed, i) for i, s in enumerate(shapes)]
    ora = [oracle_tensor(orc, m.numpy(), s, slice_p) for m, s in zip(masters, shapes)]
    keep, descs, ws, rs, p0s, ss = [], [], [], [], [], []
    for i, s in enumerate(shapes):
        n = W.numel(s)
        ot = ora[i]
        b1, w = alloc_offset(n, torch.int16, 1)
        b2, r = alloc_offset(n, torch.int16, 3)
        if n:
            w.copy_(torch.from_numpy(ot["hi"].view(np.int16)))
            r.copy_(torch.from_numpy(ot["lo"].view(np.int16)))
        if "row" in ot:
            b3, rw = alloc_offset(ot["row"].size, torch.float32, 1)
            b4, cl = alloc_offset(ot["col"].size, torch.float32, 1)
            rw.zero_(), cl.zero_()
        else:
            b3, rw = None, None
            b4, cl = alloc_offset(n, torch.float32, 1)
            cl.zero_()
        L = max(lmopt.optim_prodigy_slice_len(n, slice_p), 1)
        b5, p0 = alloc_offset(L, torch.float32, 1)
        b6, sv = alloc_offset(L, torch.float32, 1)
        keep += [b1, b2, b3, b4, b5, b6]
        d = lmopt.TensorDesc(w_bf16=w.data_ptr() if n else None, res_u16=r.data_ptr() if n else None,
                             m=rw.data_ptr() if (rw is not None and rw.numel()) else None,
                             v=cl.data_ptr() if cl.numel() else None, numel=n, ndim=len(s))
        for k, dim in enumerate(s):
            d.shape[k] = dim
        descs.append(d)
        ws.append(w), rs.append(r), p0s.append(p0), ss.append(sv)
    h = lmopt.optim_group_create(descs, lmopt.OPTIM_KIND_FACTORED)
    pd = lmopt.optim_prodigy_create(d0, beta3, slice_p)
    H = lmopt.FactoredHparams(lr=hp["lr"], beta2=hp["beta2"], decay_rate=hp["decay_rate"], eps1=hp["eps1"],
                              eps2=hp["eps2"], d=1.0, clip_threshold=hp["clip_threshold"],
                              weight_decay=hp["weight_decay"], mode=1)
    try:
        lmopt.optim_group_attach_prodigy(h, pd, [x.data_ptr() for x in p0s], [x.data_ptr() for x in ss], 1, 0)
        lrd = 0.0
        for t in range(1, steps + 1):
            bias = [W.grad_bf16(s, seed + 1, i, 0, 1e-3).float() for i, s in enumerate(shapes)]
            grads = [(bias[i] + W.grad_bf16(s, seed, i, t, 3e-4).float()).to(torch.bfloat16)
                     for i, s in enumerate(shapes)]
            lrd += hp["lr"] * st.d32
            orc.prodigy_step(st, [(ora, [W.bits16(g).reshape(-1) for g in grads], hp)], t)
            gbufs, ptrs = [], []
            for g in grads:
                b, gg = alloc_offset(g.numel(), torch.int16, 1)
                if g.numel():
                    gg.copy_(g.reshape(-1).view(torch.int16))
                gbufs.append(b)
                ptrs.append(gg.data_ptr() if g.numel() else None)
            lmopt.optim_step_factored(h, ptrs, t, H, 0)
            lmopt.optim_prodigy_end_step(pd, 0)
            torch.cuda.synchronize()
            d_gpu, _ = lmopt.optim_prodigy_get(pd)
            assert abs(d_gpu - st.d.value) <= 1e-5 * st.d.value, (t, d_gpu, st.d.value)
        assert st.d.value > d0
        for i, ot in enumerate(ora):
            if ot["hi"].size == 0:
                continue
            ref = orc.kahan_merge(ot["hi"], ot["lo"]).astype(np.float64)
            got = orc.kahan_merge(cuda_bits(ws[i]), cuda_bits(rs[i])).astype(np.float64)
            assert np.all(np.abs(got - ref) <= 1e-6 * np.abs(ref) + 2e-5 * lrd), f"tensor {i} {shapes[i]}"
            assert np.array_equal(p0s[i][:ot["p0"].size].cpu().numpy().view(np.uint32), ot["p0"].view(np.uint32))
            s_ref = ot["s"].astype(np.float64)
            err = np.abs(ss[i][:ot["s"].size].cpu().numpy().astype(np.float64) - s_ref)
            assert np.all(err <= 1e-5 * np.abs(s_ref) + 1e-5 * np.abs(s_ref).max()), f"tensor {i}: s differs"
    finally:
        lmopt.optim_group_destroy(h)
        lmopt.optim_prodigy_destroy(pd)
