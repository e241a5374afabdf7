"""Checkpoint and resume for every group kind other than NAdam u16 (covered in test_gpu_nadam.py):
k steps, copy the caller-owned state out (weights, residuals, state buffers) with the step
counter, build a new group over the copies, run the remaining steps, and compare with the same
N steps run without interruption -- bit for bit, since nothing of a step depends on anything
else than those buffers, the step counter and (for u16 groups) the scale records."""
import pytest
import torch

from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SHAPES_1D = [(5000,), (70001,), (300,)]
ADAN_HP = dict(lr=1e-3, beta1=0.02, beta2=0.08, beta3=0.01, eps=1e-8, weight_decay=0.02)
FACTORED_HP = dict(lr=1e-3, beta2=0.999, decay_rate=-0.8, eps1=1e-30, eps2=1e-30, d=1.0, clip_threshold=1.0,
                   weight_decay=0.01, mode=0)


@pytest.fixture(scope="module")
def eng():
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    return engine


def _bits_equal(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def _resume(eng, make, rebuild, attrs, shapes, hp, steps=5, k=3, seed=17):
    from memory_lean_optimizer_gb300 import lmopt
    masters = [W.master_weights(s, seed, i, device="cuda") for i, s in enumerate(shapes)]
    grads = {t: [W.grad_bf16(s, seed, i, t, 1e-3, device="cuda") for i, s in enumerate(shapes)]
             for t in range(1, steps + 1)}
    a = make(masters)
    for t in range(1, steps + 1):
        a.step(grads[t], hp)
    b = make(masters)
    for t in range(1, k + 1):
        b.step(grads[t], hp)
    torch.cuda.synchronize()
    saved = {name: [None if x is None else x.clone() for x in getattr(b, name)] for name in ("weights",) + attrs}
    step, mp = lmopt.optim_group_get_step(b.handle)
    b.close()
    c = rebuild(saved)
    lmopt.optim_group_set_step(c.handle, step, mp)
    c.step_count = step
    for t in range(k + 1, steps + 1):
        c.step(grads[t], hp)
    torch.cuda.synchronize()
    for name in ("weights",) + attrs:
        for i, (x, y) in enumerate(zip(getattr(a, name), getattr(c, name))):
            if x is not None:
                assert _bits_equal(x, y), (name, i)
    a.close()
    c.close()


def test_resume_nadam_f24(eng):
    def make(masters):
        return eng.NadamGroup.from_masters([m.clone() for m in masters], states="f24")

    def rebuild(saved):
        g = eng.NadamGroup([w.clone() for w in saved["weights"]], [r.clone() for r in saved["res"]], states="f24")
        for i in range(len(saved["m"])):
            g.m[i].copy_(saved["m"][i])
            g.v[i].copy_(saved["v"][i])
        return g
    _resume(eng, make, rebuild, ("res", "m", "v"), SHAPES_1D, dict(W.NADAM_HP, lr=1e-3))


@pytest.mark.parametrize("states", ["fp32", "f24"])
def test_resume_adan(eng, states):
    def make(masters):
        return eng.AdanGroup.from_masters([m.clone() for m in masters], states=states)

    def rebuild(saved):
        g = eng.AdanGroup([w.clone() for w in saved["weights"]], [r.clone() for r in saved["res"]], states=states)
        for i in range(len(saved["mvn"])):
            g.mvn[i].copy_(saved["mvn"][i])
            g.gprev[i].copy_(saved["gprev"][i])
        return g
    _resume(eng, make, rebuild, ("res", "mvn", "gprev"), SHAPES_1D, ADAN_HP)


def test_resume_factored(eng):
    shapes = [(64, 80), (3, 40, 72), (8, 8, 3, 3), (300,), (1000, 640)]

    def make(masters):
        return eng.FactoredGroup.from_masters([m.clone() for m in masters])

    def rebuild(saved):
        g = eng.FactoredGroup([w.clone() for w in saved["weights"]], [r.clone() for r in saved["res"]])
        for i in range(len(saved["col"])):
            if saved["row"][i] is not None:
                g.row[i].copy_(saved["row"][i])
            g.col[i].copy_(saved["col"][i])
        return g
    _resume(eng, make, rebuild, ("res", "row", "col"), shapes, FACTORED_HP)
