"""Canary bytes around every buffer a call touches.

Each weight, residual, state buffer, gradient and host image of these tests sits between two
512-byte guards filled with a known byte.  After the calls, every guard must still hold that byte
and every gradient must be unchanged, so a write past either end of a buffer (a ragged head or
tail, a vector access that runs over, a wrong stride) shows up here even without a memory checker.
Sizes sit on both sides of the vector widths (8 elements), of the small-tensor limit (4096) and of
the chunk sizes (2048..32768); buffers start either on a 16-byte boundary or at the smallest
offset each buffer accepts (2 bytes, 4 for fp32 states), which takes the element-by-element paths.
The guarded group's results must also equal those of an ordinary group stepped alongside it.
"""
import numpy as np
import pytest
import torch

from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 512
CANARY = 0xA5
SIZES = [1, 2, 3, 7, 8, 9, 15, 16, 17, 4095, 4096, 4097, 8191, 16383, 16384, 16385, 32767, 32769, 65537]
FACTORED_SHAPES = [(1,), (3,), (4097,), (1, 1), (3, 5), (17, 33), (64, 4097), (257, 129), (2, 3, 5, 7)]
ADAN_HP = dict(lr=1e-3, beta1=0.02, beta2=0.08, beta3=0.01, eps=1e-8, weight_decay=0.02)
FACTORED_HP = dict(lr=1e-3, beta2=0.999, decay_rate=-0.8, eps1=1e-30, eps2=1e-30, d=1.0, clip_threshold=1.0,
                   weight_decay=0.01, mode=0)


@pytest.fixture(scope="module")
def eng():
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    return engine


class Guarded:
    """`nbytes` bytes starting `offset` bytes past a 512-byte guard, followed by another guard."""

    def __init__(self, nbytes, offset, pinned=False):
        total = GUARD + offset + nbytes + GUARD
        if pinned:
            self.buf = torch.full((total,), CANARY, dtype=torch.uint8).pin_memory()
        else:
            self.buf = torch.full((total,), CANARY, dtype=torch.uint8, device="cuda")
        self.start, self.nbytes = GUARD + offset, nbytes

    def view(self, dtype, shape):
        return self.buf[self.start:self.start + self.nbytes].view(dtype).view(shape)

    def ptr(self):
        return self.buf.data_ptr() + self.start

    def intact(self):
        b = self.buf
        return bool((b[:self.start] == CANARY).all()) and bool((b[self.start + self.nbytes:] == CANARY).all())


def _offset(t, misaligned, at_least=0):
    return max(4 if t.element_size() == 4 else 2, at_least) if misaligned else 0


def _guarded_copy(t, misaligned, guards, at_least=0):
    g = Guarded(t.numel() * t.element_size(), _offset(t, misaligned, at_least))
    v = g.view(t.dtype, t.shape)
    v.copy_(t)
    guards.append(g)
    return v


def rehome(eng, grp, attrs, misaligned, move=None, align=None):
    """Moves the group's weights and state buffers (attribute lists `attrs`, in descriptor order;
    only those named in `move`, if given) into guarded buffers and re-creates its handle over
    them; `align` names lists whose offset must be at least so many bytes.  Returns the guards."""
    align = align or {}
    from memory_lean_optimizer_gb300 import lmopt
    torch.cuda.synchronize()
    guards = []
    names = ("weights",) + tuple(attrs)
    lists = [getattr(grp, a) for a in names]
    moved = [[t if (t is None or t.numel() == 0 or (move is not None and name not in move))
              else _guarded_copy(t, misaligned, guards, align.get(name, 0)) for t in lst]
             for name, lst in zip(names, lists)]
    descs = [eng._desc(*[ml[i] for ml in moved], moved[0][i].shape) for i in range(len(grp.weights))]
    new = lmopt.optim_group_create(descs, grp.kind)
    lmopt.optim_group_destroy(grp.handle)
    grp.handle = new
    grp.weights = moved[0]
    for a, ml in zip(attrs, moved[1:]):
        setattr(grp, a, ml)
    return guards


def guarded_grads(shapes, seed, t, misaligned, guards):
    grads, copies = [], []
    for i, s in enumerate(shapes):
        g = W.grad_bf16(s, seed, i, t, 1e-3, zero_frac=0.01, device="cuda")
        grads.append(_guarded_copy(g, misaligned, guards))
        copies.append(g)
    return grads, copies


def _bits(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def check_guards(guards, grads, copies, what):
    torch.cuda.synchronize()
    bad = [i for i, g in enumerate(guards) if not g.intact()]
    assert not bad, f"{what}: guard bytes overwritten around buffers {bad}"
    for a, b in zip(grads, copies):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{what}: a gradient was written"


def _pair(eng, cls, masters, **kw):
    return cls.from_masters([m.clone() for m in masters], **kw), cls.from_masters([m.clone() for m in masters], **kw)


@pytest.mark.parametrize("misaligned", [False, True], ids=["aligned", "misaligned"])
@pytest.mark.parametrize("variant", ["u16", "f24", "sr"])
def test_nadam_guards(eng, misaligned, variant):
    shapes = [(n,) for n in SIZES]
    seed = 81
    masters = [W.master_weights(s, seed, i, device="cuda") for i, s in enumerate(shapes)]
    hp = dict(W.NADAM_HP, lr=1e-3)
    if variant == "sr":
        hp = dict(hp, stochastic_rounding=1, seed=7)
        ws = [eng.kahan_split(m)[0] for m in masters]
        grp = eng.NadamGroup([w.clone() for w in ws], kahan=False)
        twin = eng.NadamGroup([w.clone() for w in ws], kahan=False)
    else:
        grp, twin = _pair(eng, eng.NadamGroup, masters, states=variant)
    guards = rehome(eng, grp, ("res", "m", "v"), misaligned)
    for t in range(1, 4):
        grads, copies = guarded_grads(shapes, seed, t, misaligned, guards)
        grp.step(grads, hp)
        twin.step(copies, hp)
        check_guards(guards, grads, copies, f"step {t}")
    for name in ("weights", "res", "m", "v"):
        for i, (a, b) in enumerate(zip(getattr(grp, name), getattr(twin, name))):
            if a is not None and a.numel():
                assert np.array_equal(_bits(a), _bits(b)), (name, i)
    grp.close()
    twin.close()


@pytest.mark.parametrize("states", ["u16", "f24"])
def test_nadam_guards_two_launch_group(eng, states):
    """A group too large for the one-launch step: u16 moments take the pre-pass and the update as
    two kernels; f24 moments need no pre-pass and take one kernel at any size."""
    shapes = [(50_000_001,), (4097,), (3,)]
    seed = 82
    masters = [W.master_weights(s, seed, i, device="cuda") for i, s in enumerate(shapes)]
    hp = dict(W.NADAM_HP, lr=1e-3)
    grp, twin = _pair(eng, eng.NadamGroup, masters, states=states)
    guards = rehome(eng, grp, ("res", "m", "v"), True)
    assert grp.launches(hp) == (2 if states == "u16" else 1)
    for t in range(1, 3):
        grads, copies = guarded_grads(shapes, seed, t, True, guards)
        grp.step(grads, hp)
        twin.step(copies, hp)
        check_guards(guards, grads, copies, f"step {t}")
    for name in ("weights", "res", "m", "v"):
        for a, b in zip(getattr(grp, name), getattr(twin, name)):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name
    grp.close()
    twin.close()


def test_nadam_one_launch_group_is_fused(eng):
    """The SIZES group takes the one-launch step, so the guards above cover that kernel too."""
    masters = [W.master_weights((n,), 83, i, device="cuda") for i, n in enumerate(SIZES)]
    grp = eng.NadamGroup.from_masters(masters)
    assert grp.launches(dict(W.NADAM_HP)) == 1
    grp.close()


@pytest.mark.parametrize("misaligned", [False, True], ids=["aligned", "misaligned"])
@pytest.mark.parametrize("states", ["fp32", "f24"])
def test_adan_guards(eng, misaligned, states):
    shapes = [(n,) for n in SIZES]
    seed = 84
    masters = [W.master_weights(s, seed, i, device="cuda") for i, s in enumerate(shapes)]
    grp, twin = _pair(eng, eng.AdanGroup, masters, states=states)
    guards = rehome(eng, grp, ("res", "mvn", "gprev"), misaligned, align={"mvn": 4})   # f24 bytes: 4-byte start
    for t in range(1, 4):
        grads, copies = guarded_grads(shapes, seed, t, misaligned, guards)
        grp.step(grads, ADAN_HP)
        twin.step(copies, ADAN_HP)
        check_guards(guards, grads, copies, f"step {t}")
    for name in ("weights", "res", "mvn", "gprev"):
        for i, (a, b) in enumerate(zip(getattr(grp, name), getattr(twin, name))):
            assert np.array_equal(_bits(a), _bits(b)), (name, i)
    grp.close()
    twin.close()


@pytest.mark.parametrize("misaligned", [False, True], ids=["aligned", "misaligned"])
def test_factored_guards(eng, misaligned):
    seed = 85
    masters = [W.master_weights(s, seed, i, device="cuda") for i, s in enumerate(FACTORED_SHAPES)]
    grp, twin = _pair(eng, eng.FactoredGroup, masters)
    guards = rehome(eng, grp, ("res", "row", "col"), misaligned)
    for t in range(1, 4):
        grads, copies = guarded_grads(FACTORED_SHAPES, seed, t, misaligned, guards)
        grp.step(grads, FACTORED_HP)
        twin.step(copies, FACTORED_HP)
        check_guards(guards, grads, copies, f"step {t}")
    # same kernels on the same values; the factored tests' tolerance covers any change of path
    for a, b in zip(grp.masters(), twin.masters()):
        a, b = a.double(), b.double()
        assert torch.all((a - b).abs() <= 1e-6 * b.abs() + 1e-6 * FACTORED_HP["lr"] * 3)
    grp.close()
    twin.close()


@pytest.mark.parametrize("misaligned", [False, True], ids=["aligned", "misaligned"])
def test_factored_noalloc_guards(eng, misaligned):
    from memory_lean_optimizer_gb300 import lmopt
    shape, seed = (257, 129), 86
    master = W.master_weights(shape, seed, 0, device="cuda")
    grp, twin = _pair(eng, eng.FactoredGroup, [master])
    guards = rehome(eng, grp, ("res", "row", "col"), misaligned)
    d = eng._desc(grp.weights[0], grp.res[0], grp.row[0], grp.col[0], shape)
    h = lmopt.FactoredHparams(**FACTORED_HP)
    for t in range(1, 3):
        grads, copies = guarded_grads([shape], seed, t, misaligned, guards)
        lmopt.optim_step_factored_noalloc(d, grads[0].data_ptr(), t, h, torch.cuda.current_stream().cuda_stream)
        twin.step(copies, FACTORED_HP)
        check_guards(guards, grads, copies, f"step {t}")
    a, b = grp.masters()[0].double(), twin.masters()[0].double()
    assert torch.all((a - b).abs() <= 1e-6 * b.abs() + 1e-6 * FACTORED_HP["lr"] * 2)
    grp.close()
    twin.close()


@pytest.mark.parametrize("n", [1, 7, 9, 4097, 16385, 65537])
@pytest.mark.parametrize("misaligned", [False, True], ids=["aligned", "misaligned"])
def test_codec_and_kahan_guards(eng, n, misaligned):
    from memory_lean_optimizer_gb300 import lmopt
    stream = torch.cuda.current_stream().cuda_stream
    guards = []
    off2, off4 = (2, 4) if misaligned else (0, 0)
    master = W.master_weights((n,), 87, 0, device="cuda")
    gx, ghi, glo, gout = Guarded(4 * n, off4), Guarded(2 * n, off2), Guarded(2 * n, off2), Guarded(4 * n, off4)
    guards += [gx, ghi, glo, gout]
    gx.view(torch.float32, (n,)).copy_(master)
    lmopt.optim_kahan_split(gx.ptr(), ghi.ptr(), glo.ptr(), n, stream)
    lmopt.optim_kahan_merge(ghi.ptr(), glo.ptr(), gout.ptr(), n, stream)
    torch.cuda.synchronize()
    assert torch.equal(gout.view(torch.int32, (n,)), gx.view(torch.int32, (n,)))
    for signed in (True, False):
        x = master if signed else master.abs()
        gin, gcodes, gscale, gback = Guarded(4 * n, off4), Guarded(2 * n, off2), Guarded(4, off4), Guarded(4 * n, off4)
        guards += [gin, gcodes, gscale, gback]
        gin.view(torch.float32, (n,)).copy_(x)
        lmopt.state_pack_u16(gin.ptr(), gcodes.ptr(), gscale.ptr(), n, signed, stream)
        lmopt.state_unpack_u16(gcodes.ptr(), gscale.ptr(), gback.ptr(), n, signed, stream)
    torch.cuda.synchronize()
    assert all(g.intact() for g in guards)


def test_offload_host_image_guards(eng):
    """The per-group offload calls copy exactly the layout's bytes in and out of a guarded host
    image; weights, residuals and moment codes equal those of a group stepped on the device."""
    from memory_lean_optimizer_gb300 import lmopt
    shapes = [(n,) for n in SIZES]
    seed = 88
    masters = [W.master_weights(s, seed, i, device="cuda") for i, s in enumerate(shapes)]
    hp = dict(W.NADAM_HP, lr=1e-3)
    grp, twin = _pair(eng, eng.NadamGroup, masters)
    guards = rehome(eng, grp, ("res", "m", "v"), True, move=("weights",))   # weights guarded on the device
    total, offs = lmopt.optim_offload_layout(grp.handle, len(shapes))
    image = Guarded(total, 0, pinned=True)
    lmopt.optim_group_attach_host(grp.handle, image.ptr(), total)
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    for t in range(1, 4):
        grads, copies = guarded_grads(shapes, seed, t, True, guards)
        grp.prefetch(cin)
        grp.step(grads, hp)
        grp.writeback(cout)
        twin.step(copies, hp)
        eng.OffloadEngine.sync_library_ring()
        check_guards(guards, grads, copies, f"step {t}")
        assert image.intact(), f"step {t}: host image guard overwritten"
    img = image.buf[image.start:image.start + total].numpy()
    for i, n in enumerate(SIZES):
        assert torch.equal(grp.weights[i].view(torch.int16), twin.weights[i].view(torch.int16))
        for k, ref in enumerate((twin.res[i], twin.m[i], twin.v[i])):
            nb = ref.numel() * ref.element_size()
            assert np.array_equal(img[offs[i][k]:offs[i][k] + nb], _bits(ref)), (i, k)
    grp.close()
    twin.close()
