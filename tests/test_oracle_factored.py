"""Pins of the oracle's factored second-moment step (Adafactor; Prodigy's factored variant).

The step follows the printed fused Adafactor step ("Fused backward pass" commit,
library/adafactor_fused.py, adafactor_step_param): row/column EMAs of g^2+eps1 over the last
two dims, the rank-1 reconstruction of the Adafactor paper, RMS update clipping, decoupled
decay, beta1 = 0 with no exp_avg ("more VRAM savings: no first moment and factored second
moment", prodigy PR #25).  The pins: torch.optim.Adafactor (library routine) in the settings
where it computes the same thing, the rank-1 case where the factored estimate is exact, the
1-D step-1 sign, clipping to exactly the threshold, and a zero gradient.
"""
import numpy as np
import pytest
import torch

from test_oracle_nadam import bf16_bits, bits_to_f32

HP = dict(lr=1e-2, beta2=0.999, decay_rate=-0.8, eps1=1e-30, eps2=1e-30, d=1.0,
          clip_threshold=1.0, weight_decay=0.0, mode=0)


def make(orc, shape, w0):
    hi, lo = orc.kahan_split(w0.astype(np.float32).reshape(-1))
    fac, B, R, C = orc.factored_dims(shape)
    t = dict(hi=hi, lo=lo, shape=shape)
    if fac:
        t["row"] = np.zeros(B * R, np.float32)
        t["col"] = np.zeros(B * C, np.float32)
    else:
        t["V"] = np.zeros(hi.size, np.float32)
    return t


def run(orc, shape, w0, grads, hp):
    t = make(orc, shape, w0)
    dens = []
    for step, g in enumerate(grads, start=1):
        _, d = orc.factored_group_step([t], [g.reshape(-1)], step, hp)
        dens.append(d[0])
    return orc.kahan_merge(t["hi"], t["lo"]).reshape(shape), t, dens


@pytest.mark.parametrize("shape", [(96, 80), (40, 200), (6, 5, 3, 3), (300,)])
@pytest.mark.parametrize("wd", [0.0, 0.05])
def test_matches_torch_adafactor(orc, shape, wd):
    """torch.optim.Adafactor uses alpha = max(eps2, RMS(p)) min(lr, 1/sqrt t) and clamps V at
    eps1^2 instead of adding eps1; with eps2 = 1 > RMS(p), lr < 1/sqrt(t) and nonzero g the two
    compute the same update, clip threshold d included."""
    rng = np.random.default_rng(20)
    steps = 6
    w0 = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    grads = [bf16_bits(rng.standard_normal(shape) * (1 + 3 * (k % 2))) for k in range(steps)]
    for g in grads:
        g[bits_to_f32(g) == 0] = bf16_bits(np.array([0.5]))[0]
    hp = dict(HP, eps1=0.0, weight_decay=wd, clip_threshold=1.0)
    ours, _, dens = run(orc, shape, w0, grads, hp)
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.Adafactor([p], lr=hp["lr"], beta2_decay=-0.8, eps=(1e-30, 1.0), d=1.0,
                                weight_decay=wd, foreach=False)
    for g in grads:
        p.grad = torch.from_numpy(bits_to_f32(g).reshape(shape).copy())
        opt.step()
    ref = p.detach().numpy()
    d_ours = ours.astype(np.float64) - w0
    d_ref = ref.astype(np.float64) - w0
    tol = 2e-5 * hp["lr"] * steps + 4 * np.spacing(np.abs(w0)).astype(np.float64)
    if wd:
        tol = tol + steps * np.abs(w0).astype(np.float64) * 2.0 ** -24
    assert np.all(np.abs(d_ours - d_ref) <= tol), np.max(np.abs(d_ours - d_ref) - tol)
    assert any(d > 1.0 for d in dens) and any(d == 1.0 for d in dens)   # both branches of the clip


def _rank1_grad(rng, B, R, C):
    a = rng.choice([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0], size=(B, R, 1))
    b = rng.choice([-4.0, -1.0, -0.25, 0.25, 1.0, 4.0], size=(B, 1, C))
    return (a * b).astype(np.float32)          # every product is a power of two: exact in bf16


@pytest.mark.parametrize("shape", [(64, 48), (4, 6, 3, 3), (1, 33)])
def test_rank1_gives_sign(orc, shape):
    """g^2 = a b^T is rank 1, so R C / mean(R) = g^2 exactly: u = sign(g), RMS(u) = 1, and with
    clip = 1 every step moves w by -lr sign(g) (constant g keeps the EMAs fixed)."""
    rng = np.random.default_rng(21)
    fac, B, R, C = orc.factored_dims(shape)
    g32 = _rank1_grad(rng, B, R, C).reshape(shape)
    g = bf16_bits(g32)
    assert np.array_equal(bits_to_f32(g).reshape(shape), g32)
    lr = 2.0 ** -10
    hp = dict(HP, lr=lr, eps1=0.0)
    t = make(orc, shape, np.zeros(shape, np.float32))
    for step in range(1, 6):
        orc.factored_group_step([t], [g.reshape(-1)], step, hp)
        w = orc.kahan_merge(t["hi"], t["lo"]).reshape(shape).astype(np.float64)
        expect = -step * lr * np.sign(g32)
        assert np.all(np.abs(w - expect) <= step * 8 * np.spacing(np.float32(lr)))


def test_prodigy_mode_rank1_clipped(orc):
    """Prodigy mode, d = 1, constant beta2: at t = 1, V^ = (1-beta2) g^2 (+eps2), so
    RMS(u) = 1/sqrt(1-beta2) > clip = 1 and clipping brings the step back to -lr sign(g)."""
    rng = np.random.default_rng(22)
    shape = (32, 24)
    g32 = _rank1_grad(rng, 1, *shape).reshape(shape)
    g = bf16_bits(g32)
    lr = 2.0 ** -10
    hp = dict(HP, lr=lr, mode=1, beta2=0.99, eps2=1e-30)
    w, _, dens = run(orc, shape, np.zeros(shape, np.float32), [g], hp)
    assert abs(dens[0] - 1 / np.sqrt(1 - 0.99)) < 1e-4 * dens[0]
    assert np.all(np.abs(w + lr * np.sign(g32)) <= 8 * np.spacing(np.float32(lr)))


def test_vector_step1_sign(orc):
    rng = np.random.default_rng(23)
    n = 5000
    g32 = rng.standard_normal(n).astype(np.float32) * 1e-2
    g = bf16_bits(g32)
    gf = bits_to_f32(g)
    keep = gf != 0
    lr = 2.0 ** -12
    w, _, dens = run(orc, (n,), np.zeros(n, np.float32), [g], dict(HP, lr=lr))
    assert np.all(np.abs(w[keep] + lr * np.sign(gf[keep])) <= 8 * np.spacing(np.float32(lr)))
    assert np.all(w[~keep] == 0)


@pytest.mark.parametrize("shape", [(64, 64), (500,)])
def test_clipped_rms_equals_threshold(orc, shape):
    """After clipping, RMS(update / lr) <= clip, with equality whenever clipping is active."""
    rng = np.random.default_rng(24)
    g32 = (rng.standard_normal(shape) * 1e-3).astype(np.float32)
    g32.reshape(-1)[::37] *= 50.0                     # spikes the factored estimate misses
    g = bf16_bits(g32)
    lr, clip = 2.0 ** -10, 0.5
    w, _, dens = run(orc, shape, np.zeros(shape, np.float32), [g], dict(HP, lr=lr, clip_threshold=clip))
    assert dens[0] > 1.0
    rms = np.sqrt(np.mean((w.astype(np.float64) / lr) ** 2))
    assert abs(rms - clip) < 1e-5 * clip
    w2, _, dens2 = run(orc, shape, np.zeros(shape, np.float32), [g], dict(HP, lr=lr, clip_threshold=1e6))
    assert dens2[0] == 1.0
    assert np.sqrt(np.mean((w2.astype(np.float64) / lr) ** 2)) <= 1e6


@pytest.mark.parametrize("shape", [(16, 20), (2, 2, 3, 3), (77,)])
def test_zero_grad_is_identity(orc, shape):
    rng = np.random.default_rng(25)
    w0 = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    z = np.zeros(shape, np.uint16)
    w, t, _ = run(orc, shape, w0, [z, z, z], dict(HP, eps1=1e-30))
    assert np.array_equal(w, w0)


@pytest.mark.parametrize("shape", [(0, 64), (5, 0), (0, 3, 3, 3), (0,)])
def test_empty_tensor_leaves_state(orc, shape):
    """A tensor without elements has no gradient: its state stays as it was (no 0/0 mean) and the
    other tensors of the group step as they would alone."""
    rng = np.random.default_rng(26)
    other = (rng.standard_normal((12, 8)) * 0.02).astype(np.float32)
    g_other = bf16_bits(rng.standard_normal((12, 8)) * 1e-3)
    empty = make(orc, shape, np.zeros(shape, np.float32))
    for name in ("row", "col", "V"):
        if name in empty:
            empty[name][:] = 0.5
    t_alone = make(orc, (12, 8), other)
    t_group = make(orc, (12, 8), other)
    orc.factored_group_step([t_alone], [g_other.reshape(-1)], 1, HP)
    _, dens = orc.factored_group_step([empty, t_group], [np.zeros(0, np.uint16), g_other.reshape(-1)], 1, HP)
    for name in ("row", "col", "V"):
        if name in empty:
            assert np.all(empty[name] == 0.5)
    assert dens[0] == 1.0
    assert np.array_equal(t_group["hi"], t_alone["hi"]) and np.array_equal(t_group["lo"], t_alone["lo"])


def test_zero_row_with_eps1_zero_is_flagged(orc):
    """eps1 = 0 and an all-zero gradient row: that row's R is 0, its factor rsqrt(0) is infinite
    and 0 * inf is NaN, so the row's update -- and through the RMS clip, whose clamp(min=1) keeps
    a NaN, the whole tensor -- is NaN.  The oracle reports this (non-finite weights) instead of
    hiding it; with eps1 > 0 the same gradient gives finite weights and leaves the zero row's
    weights unchanged."""
    rng = np.random.default_rng(27)
    shape = (8, 12)
    w0 = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    g = rng.standard_normal(shape).astype(np.float32)
    g[3, :] = 0.0
    gb = bf16_bits(g)
    w_nan, _, _ = run(orc, shape, w0, [gb], dict(HP, eps1=0.0))
    assert np.isnan(w_nan[3]).all() and np.isnan(w_nan).all()
    w_ok, _, _ = run(orc, shape, w0, [gb], dict(HP, eps1=1e-30))
    assert np.isfinite(w_ok).all() and np.array_equal(w_ok[3], w0[3])
