"""GPU parity of the factored second-moment step (Adafactor / Prodigy, beta1 = 0) against the
oracle, through the C ABI.

The oracle sums rows, columns and squares in double; the kernels use fp32 trees (and compensated
sums across tiles), so R, C and the clip divisor agree to a few fp32 roundings, not bit for bit.
Tolerances, derived from that:
  R, C states      : 1e-6 relative  (sums of positive terms: a tree of n terms rounds at most
                     ceil(log2 n) times per term, 14 * 2^-24 = 8.3e-7 for 10240 columns, plus the
                     EMA's two roundings; the cases here reach 2.4e-7)
  fp32 masters     : |w - w_ref| <= 1e-6 |w_ref| + 1e-6 (lr d steps + sum_k |update_k|)  (the
                     kernels' update is within a few ulps of the oracle's -- the statistics above,
                     and the per-tensor scale fl(u fl(lr/den)) for fl(fl(u/den) lr) -- and single
                     elements' updates reach several times lr d; plus one rounding of w)
"""
import numpy as np
import pytest
import torch

from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta2=0.999, decay_rate=-0.8, eps1=1e-30, eps2=1e-30, d=1.0, clip_threshold=1.0,
          weight_decay=0.0, mode=0)


@pytest.fixture(scope="module")
def eng():
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    return engine


class OracleFactored:
    def __init__(self, orc, masters, shapes, kahan=True):
        self.orc = orc
        self.t = []
        for x, s in zip(masters, shapes):
            x = np.ascontiguousarray(x, np.float32).reshape(-1)
            hi, lo = orc.kahan_split(x) if kahan else (orc.round_bf16(x), None)
            fac, B, R, C = orc.factored_dims(s)
            d = dict(hi=hi, lo=lo, shape=s)
            if fac:
                d["row"] = np.zeros(B * R, np.float32)
                d["col"] = np.zeros(B * C, np.float32)
            else:
                d["V"] = np.zeros(x.size, np.float32)
            self.t.append(d)
        self.steps = 0

    def step(self, grads, hp):
        self.steps += 1
        before = [self._master(t) for t in self.t]
        self.orc.factored_group_step(self.t, grads, self.steps, hp)
        for t, b in zip(self.t, before):   # sum over the steps of each element's |update|
            if b is not None:
                t["moved"] = t.get("moved", 0.0) + np.abs(self._master(t) - b)

    def _master(self, t):
        return self.orc.kahan_merge(t["hi"], t["lo"]).astype(np.float64) if t["lo"] is not None else None


def compare(ora, grp, hp, steps, kahan=True, upd_tol=1e-6):
    masters = grp.masters() if kahan else None
    for i, ot in enumerate(ora.t):
        if ot["hi"].size == 0:
            continue
        if kahan:
            ref = ora.orc.kahan_merge(ot["hi"], ot["lo"]).astype(np.float64)
            got = masters[i].cpu().numpy().reshape(-1).astype(np.float64)
            tol = 1e-6 * np.abs(ref) + upd_tol * (hp["lr"] * hp.get("d", 1.0) * steps + ot.get("moved", 0.0))
            bad = np.abs(got - ref) > tol
            assert not bad.any(), f"tensor {i} {ot['shape']}: {bad.sum()} masters out of tolerance, " \
                                  f"max excess {np.max(np.abs(got - ref) - tol):.3e}"
        else:
            ref = (ot["hi"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            got = grp.weights[i].float().cpu().numpy().reshape(-1).astype(np.float64)
            step = np.abs(ref) * 2.0 ** -7 + 1e-30
            assert np.all(np.abs(got - ref) <= step), f"tensor {i}: bf16 weights differ by more than one step"
            assert np.mean(got != ref) < 1e-3
        if "row" in ot:
            for name, st in (("row", grp.row[i]), ("col", grp.col[i])):
                r = ot[name].astype(np.float64)
                gv = st.cpu().numpy().astype(np.float64)
                assert np.all(np.abs(gv - r) <= 1e-6 * np.abs(r) + 1e-37), f"tensor {i}: {name} state differs"
        else:
            r = ot["V"].astype(np.float64)
            gv = grp.col[i].cpu().numpy().astype(np.float64)
            assert np.all(np.abs(gv - r) <= 1e-6 * np.abs(r) + 1e-37), f"tensor {i}: V state differs"


def run_parity(orc, eng, shapes, steps, hp, seed=0, g_std=1e-3, kahan=True, scale_rows=False, upd_tol=1e-6):
    masters = [W.master_weights(s, seed, i) for i, s in enumerate(shapes)]
    ora = OracleFactored(orc, [m.numpy() for m in masters], shapes, kahan=kahan)
    if kahan:
        grp = eng.FactoredGroup.from_masters([m.cuda() for m in masters])
    else:
        grp = eng.FactoredGroup([m.cuda().to(torch.bfloat16) for m in masters], kahan=False)
    for t in range(1, steps + 1):
        grads = []
        for i, s in enumerate(shapes):
            g = W.grad_bf16(s, seed, i, t, g_std)
            if scale_rows and len(s) >= 2:      # uneven row/column scales exercise clipping
                g = (g.float() * torch.linspace(0.1, 3.0, s[-1])).to(torch.bfloat16)
            grads.append(g)
        ora.step([W.bits16(g).reshape(-1) for g in grads], hp)
        grp.step([g.cuda() for g in grads], hp)
    torch.cuda.synchronize()
    compare(ora, grp, hp, steps, kahan=kahan, upd_tol=upd_tol)
    from memory_lean_optimizer_gb300 import lmopt
    assert lmopt.optim_query_nonfinite(grp.handle) == 0
    return ora, grp


# (45, 50, 3, 3): 2250 small matrices, one full CTA of 2048 and a ragged one (202: no 128-bit
# staging); (600, 2, 2): the generic small-matrix path over three sub-batches
SHAPES = [(64, 80), (300, 257), (1000, 640), (3, 40, 72), (1, 300), (300, 1), (4, 6, 3, 3), (32, 16, 3, 3),
          (2, 2), (1280,), (77,), (5000,), (45, 50, 3, 3), (600, 2, 2)]


@pytest.mark.parametrize("mode", [0, 1])
def test_mixed_shapes(orc, eng, mode):
    hp = dict(HP, mode=mode, beta2=0.99)
    run_parity(orc, eng, SHAPES, 4, hp, seed=1, scale_rows=True)


def test_prodigy_mode_fixed_d(orc, eng):
    """Prodigy mode with a fixed d != 1: the update's numerator d g and the step size d lr on every
    tensor class (wide, batched, 3x3, small, 1-D), clipped and unclipped.  The kernels multiply
    each element's update by d before its square is summed and before the clip, as the oracle
    does, so the tolerance is the one of Adafactor mode."""
    hp = dict(HP, mode=1, beta2=0.99, d=0.37, weight_decay=0.02)
    run_parity(orc, eng, SHAPES, 3, hp, seed=8, scale_rows=True)
    run_parity(orc, eng, SHAPES[:6], 2, dict(hp, clip_threshold=1e3), seed=9)


def test_weight_decay_and_clip_threshold(orc, eng):
    hp = dict(HP, weight_decay=0.05, clip_threshold=0.5)
    run_parity(orc, eng, SHAPES[:8], 3, hp, seed=2)


def test_sdxl_like_shapes_reduced(orc, eng):
    """The SDXL-like tensor kinds at their real sizes: a 10240x1280 and a 1280x5120 linear, a
    1280x1280 3x3 conv, 2048-wide linears and 1-D norms/biases."""
    shapes = [(10240, 1280), (1280, 5120), (1280, 2048), (640, 640), (1280, 1280, 3, 3), (320, 320, 3, 3),
              (1280,), (640,)]
    hp = dict(HP, lr=2e-6, eps1=1e-30)
    run_parity(orc, eng, shapes, 2, hp, seed=3, g_std=1e-4)


def test_no_residual(orc, eng):
    # (16, 32, 3, 3): 512 whole 3x3 matrices take the specialised path without a residual
    run_parity(orc, eng, [(96, 130), (8, 8, 3, 3), (16, 32, 3, 3), (500,)], 3, dict(HP), seed=4, kahan=False)


def test_rank1_sign_on_gpu(eng):
    """Rank-1 g^2 with eps1 = 0: every step moves w by exactly -lr sign(g) (to a few ulps)."""
    rng = np.random.default_rng(5)
    R, C = 96, 72
    a = rng.choice([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0], size=(R, 1))
    b = rng.choice([-4.0, -1.0, -0.25, 0.25, 1.0, 4.0], size=(1, C))
    g32 = torch.from_numpy((a * b).astype(np.float32))
    lr = 2.0 ** -10
    grp = eng.FactoredGroup.from_masters([torch.zeros(R, C, device="cuda")])
    for t in range(1, 4):
        grp.step([g32.to(torch.bfloat16).cuda()], dict(HP, lr=lr, eps1=0.0))
    w = grp.masters()[0].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(w + 3 * lr * np.sign(g32.numpy())) <= 3 * 8 * np.spacing(np.float32(lr)))


def test_factored_validation(eng):
    from memory_lean_optimizer_gb300 import lmopt
    grp = eng.FactoredGroup.from_masters([torch.zeros(16, 16, device="cuda")])
    g = torch.zeros(16, 16, dtype=torch.bfloat16, device="cuda")
    bad = lmopt.FactoredHparams(lr=1e-3, clip_threshold=0.0)
    with pytest.raises(lmopt.LmoptError):
        lmopt.optim_step_factored(grp.handle, [g.data_ptr()], 1, bad, 0)
    with pytest.raises(lmopt.LmoptError):
        lmopt.optim_step_nadam_kahan(grp.handle, [g.data_ptr()], 1, lmopt.NadamHparams(lr=1e-3, beta1=0.9, beta2=0.99), 0)


def test_two_waves_on_two_streams(orc, eng):
    """A group larger than one wave (two 4096x6144 linears, 100 MB of gradients, and a 3x3 conv):
    its waves run on the caller's stream and the group's second stream."""
    shapes = [(4096, 6144), (4096, 6144), (640, 640, 3, 3), (1280,)]
    run_parity(orc, eng, shapes, 2, dict(HP, lr=2e-6), seed=7, g_std=1e-4)


def test_misaligned_buffers_and_empty_tensors(orc, eng):
    """Weights, residuals, gradients and states 2 or 4 bytes (not 16) aligned take the
    element-by-element paths; empty tensors (no rows, no columns, no elements) are left alone."""
    from helpers import alloc_offset, cuda_bits
    from memory_lean_optimizer_gb300 import lmopt
    shapes = [(96, 64), (40, 50, 3, 3), (700,), (0, 64), (5, 0), (0,), (33, 40)]
    seed, steps, hp = 8, 3, dict(HP)
    masters = [W.master_weights(s, seed, i) for i, s in enumerate(shapes)]
    ora = OracleFactored(orc, [m.numpy() for m in masters], shapes)
    keep, descs, ws, rs, rows, cols = [], [], [], [], [], []
    for i, s in enumerate(shapes):
        n = W.numel(s)
        ot = ora.t[i]
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
        keep += [b1, b2, b3, b4]
        d = lmopt.TensorDesc(w_bf16=w.data_ptr() if n else None, res_u16=r.data_ptr() if n else None,
                             m=rw.data_ptr() if (rw is not None and rw.numel()) else None,
                             v=cl.data_ptr() if cl.numel() else None, numel=n, ndim=len(s))
        for k, dim in enumerate(s):
            d.shape[k] = dim
        descs.append(d)
        ws.append(w), rs.append(r), rows.append(rw), cols.append(cl)
    h = lmopt.optim_group_create(descs, lmopt.OPTIM_KIND_FACTORED)
    H = lmopt.FactoredHparams(lr=hp["lr"], beta2=hp["beta2"], decay_rate=hp["decay_rate"], eps1=hp["eps1"],
                              eps2=hp["eps2"], d=hp["d"], clip_threshold=hp["clip_threshold"],
                              weight_decay=hp["weight_decay"], mode=hp["mode"])
    try:
        for t in range(1, steps + 1):
            grads = [W.grad_bf16(s, seed, i, t, 1e-3) for i, s in enumerate(shapes)]
            ora.step([W.bits16(g).reshape(-1) for g in grads], hp)
            gbufs, ptrs = [], []
            for g in grads:
                b, gg = alloc_offset(g.numel(), torch.int16, 1)
                if g.numel():
                    gg.copy_(g.reshape(-1).view(torch.int16))
                gbufs.append(b)
                ptrs.append(gg.data_ptr() if g.numel() else None)
            lmopt.optim_step_factored(h, ptrs, t, H, 0)
            torch.cuda.synchronize()
        for i, ot in enumerate(ora.t):
            if ot["hi"].size:
                ref = orc.kahan_merge(ot["hi"], ot["lo"]).astype(np.float64)
                got = orc.kahan_merge(cuda_bits(ws[i]), cuda_bits(rs[i])).astype(np.float64)
                tol = 1e-6 * np.abs(ref) + 1e-6 * hp["lr"] * steps
                assert np.all(np.abs(got - ref) <= tol), f"tensor {i} {shapes[i]}: masters differ"
            if "row" in ot:
                for st, r in ((rows[i], ot["row"]), (cols[i], ot["col"])):
                    gv = st.cpu().numpy().astype(np.float64)
                    assert np.all(np.abs(gv - r) <= 1e-6 * np.abs(r) + 1e-37), f"tensor {i}: state differs"
            else:
                gv = cols[i].cpu().numpy().astype(np.float64)
                assert np.all(np.abs(gv - ot["V"]) <= 1e-6 * np.abs(ot["V"]) + 1e-37), f"tensor {i}: V differs"
    finally:
        lmopt.optim_group_destroy(h)


def test_zero_row_with_eps1_zero_is_nan_like_the_oracle(orc, eng):
    """eps1 = 0 and an all-zero gradient row (a wide matrix, and one row of one 3x3 matrix): the
    row's factor is infinite, 0 * inf is NaN, and the clip's clamp keeps the NaN RMS, so every
    weight of both tensors is NaN -- in the oracle and in the kernels alike."""
    shapes = [(40, 64), (4, 2, 3, 3)]
    hp = dict(HP, eps1=0.0)
    masters = [W.master_weights(s, 11, i) for i, s in enumerate(shapes)]
    ora = OracleFactored(orc, [m.numpy() for m in masters], shapes)
    grp = eng.FactoredGroup.from_masters([m.cuda() for m in masters])
    grads = [W.grad_bf16(s, 11, i, 1, 1e-3) for i, s in enumerate(shapes)]
    grads[0][5, :] = 0
    grads[1][2, 1, 0, :] = 0
    ora.step([W.bits16(g).reshape(-1) for g in grads], hp)
    grp.step([g.cuda() for g in grads], hp)
    torch.cuda.synchronize()
    for i, got in enumerate(grp.masters()):
        ref = orc.kahan_merge(ora.t[i]["hi"], ora.t[i]["lo"])
        assert np.isnan(ref).all(), f"tensor {i}: the oracle should report NaN"
        assert np.isnan(got.cpu().numpy()).all(), f"tensor {i}: the kernels should report NaN"
    from memory_lean_optimizer_gb300 import lmopt
    # the wide matrix's 1 tile and the small-matrix tensor's 1 block stored non-finite weights
    assert lmopt.optim_query_nonfinite(grp.handle) == 2
    grp.close()


@pytest.mark.parametrize("mode", [0, 1])
def test_degenerate_gradients(orc, eng, mode):
    """Degenerate gradients on every tensor class, 5 steps, against the oracle with the tolerances
    above: all zeros for two steps then normal (state EMAs of eps1 or eps2 alone), bf16
    subnormals (squares underflow), magnitudes near 1e14 (sums of squares near 1e32; the kernels
    sum in fp32, so magnitudes whose row or column sums pass the fp32 limit are out of their
    range while the oracle's double sums are not), two scales 27 decades apart, sign flips."""
    from test_gpu_nadam import _degenerate_grad
    kinds = ["zero_then_normal", "subnormal", "large", "two_scales", "sign_flip"]
    shapes = [(64, 80), (3, 40, 72), (8, 8, 3, 3), (300,), (1000, 640)]
    cases = [(k, s) for k in kinds for s in shapes]
    hp = dict(HP, mode=mode, weight_decay=0.01)
    if mode == 1:
        hp = dict(hp, beta2=0.99, d=0.37)
    seed = 93
    masters = [W.master_weights(s, seed, i) for i, (_, s) in enumerate(cases)]
    ora = OracleFactored(orc, [m.numpy() for m in masters], [s for _, s in cases])
    grp = eng.FactoredGroup.from_masters([m.cuda() for m in masters])
    for t in range(1, 6):
        grads = []
        for i, (k, s) in enumerate(cases):
            g = _degenerate_grad(k, W.numel(s), t, seed + i)
            if k == "large":
                g = (g.float() * 1e-4).to(torch.bfloat16)     # near 1e14
            grads.append(g.reshape(s))
        ora.step([W.bits16(g).reshape(-1) for g in grads], hp)
        grp.step([g.cuda() for g in grads], hp)
    torch.cuda.synchronize()
    compare(ora, grp, hp, 5)
    from memory_lean_optimizer_gb300 import lmopt
    assert lmopt.optim_query_nonfinite(grp.handle) == 0
    grp.close()
