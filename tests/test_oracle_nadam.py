"""Pins of the oracle's NAdam(W)/Adam step with the Kahan residual and the u16 states.

The pages recommend NAdam (Nesterov momentum) and its W variant with decoupled weight decay,
without printing a formula ("Amazing Flux FFT quality on a 5090", sd-scripts PR #2187, first
post).  The oracle takes Dozat's NAdam with the momentum-decay schedule; these tests pin it to
closed forms and to torch.optim's Adam, AdamW and NAdam (library routines), using tensors of
4096 or fewer elements, which keep fp32 moments (second post of the same page).
"""
import numpy as np
import pytest
import torch

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, wd_mode=0, nesterov=1,
          momentum_decay=0.004)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def make_tensor(orc, w0: np.ndarray, small: bool):
    hi, lo = orc.kahan_split(w0.astype(np.float32))
    n = w0.size
    if small:
        return dict(hi=hi, lo=lo, m=np.zeros(n, np.float32), v=np.zeros(n, np.float32))
    return dict(hi=hi, lo=lo, m=np.full(n, 32768, np.uint16), v=np.zeros(n, np.uint16))


def run_oracle(orc, w0, grads, hp, small=True):
    t = make_tensor(orc, w0, small)
    st = orc.NadamState(1)
    for step, g in enumerate(grads, start=1):
        orc.nadam_group_step([t], [g], st, step, hp)
    return orc.kahan_merge(t["hi"], t["lo"]), t, st


@pytest.mark.parametrize("n", [1000, 50_000])
def test_adam_step1_is_lr_sign(orc, n):
    """Adam at t=1 with eps=0: m/sqrt(v) after bias correction is sign(g), so w1 - w0 = -lr sign(g)."""
    rng = np.random.default_rng(10)
    g = bf16_bits(rng.standard_normal(n) * 1e-3)
    g[bits_to_f32(g) == 0] = bf16_bits(np.array([1e-3]))[0]
    hp = dict(HP, eps=0.0, nesterov=0, lr=3.5e-6)
    w1, _, _ = run_oracle(orc, np.zeros(n, np.float32), [g], hp, small=n <= 4096)
    lr = np.float32(hp["lr"])
    ulp = np.spacing(lr)
    assert np.all(np.abs(w1.astype(np.float64) + float(lr) * np.sign(bits_to_f32(g))) <= 4 * ulp)


def test_nadam_step1_closed_form(orc):
    rng = np.random.default_rng(11)
    n = 3000
    g = bf16_bits(rng.standard_normal(n) * 1e-3)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    hp = dict(HP, lr=1e-2)
    w1, _, _ = run_oracle(orc, w0, [g], hp)
    b1, b2, psi, eps = 0.9, 0.999, 0.004, 1e-8
    mu1 = b1 * (1 - 0.5 * 0.96 ** (1 * psi))
    mu2 = b1 * (1 - 0.5 * 0.96 ** (2 * psi))
    gd = bits_to_f32(g).astype(np.float64)
    # m1 = (1-b1) g, v1 = (1-b2) g^2; NAdam's bias-corrected Nesterov numerator at t=1
    num = (1 - mu1) / (1 - mu1) * gd + mu2 / (1 - mu1 * mu2) * (1 - b1) * gd
    den = np.abs(gd) * np.sqrt(1 - b2) / np.sqrt(1 - b2) + eps
    expect = -hp["lr"] * num / den
    got = w1.astype(np.float64) - w0
    tol = 2e-6 * np.abs(expect) + 2 * np.spacing(np.abs(w0)).astype(np.float64)
    assert np.all(np.abs(got - expect) <= tol)


def _torch_traj(opt_cls, w0, grads, **kw):
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = opt_cls([p], **kw)
    for g in grads:
        p.grad = torch.from_numpy(bits_to_f32(g).copy())
        opt.step()
    return p.detach().numpy()


@pytest.mark.parametrize("variant", ["adam", "adamw", "nadam", "nadamw"])
def test_matches_torch_optim(orc, variant):
    """fp32 moments + Kahan (an exact fp32 master) reproduce torch.optim within fp32 rounding."""
    rng = np.random.default_rng(12)
    n, steps = 4096, 10
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = [bf16_bits(rng.standard_normal(n) * 1e-3) for _ in range(steps)]
    wd = 0.1 if variant.endswith("w") else 0.0
    hp = dict(HP, lr=1e-3, weight_decay=wd, wd_mode=1 if wd else 0, nesterov=variant.startswith("n"))
    ours, _, _ = run_oracle(orc, w0, grads, hp)
    if variant == "adam":
        ref = _torch_traj(torch.optim.Adam, w0, grads, lr=1e-3, betas=(0.9, 0.999), eps=1e-8)
    elif variant == "adamw":
        ref = _torch_traj(torch.optim.AdamW, w0, grads, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=wd)
    else:
        ref = _torch_traj(torch.optim.NAdam, w0, grads, lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                          momentum_decay=0.004, weight_decay=wd, decoupled_weight_decay=bool(wd))
    d_ours = ours.astype(np.float64) - w0
    d_ref = ref.astype(np.float64) - w0
    # rounding-order differences are a few ulps of each step's update (size ~lr) plus the
    # weight's own rounding; the net displacement can be small through cancellation
    tol = 1e-6 * hp["lr"] * steps + 4 * np.spacing(np.abs(w0)).astype(np.float64)
    if wd:
        # torch multiplies by fp32(1 - lr wd), whose rounding (up to 2^-25 near 1) is a large
        # relative error of the decay itself; the oracle subtracts fp32(lr wd) * w instead
        tol = tol + steps * np.abs(w0).astype(np.float64) * 2.0 ** -24
    assert np.all(np.abs(d_ours - d_ref) <= tol), np.max(np.abs(d_ours - d_ref) - tol)


def test_kahan_equals_fp32_master(orc):
    """Given equal moments the Kahan pair (hi, lo) is exactly the fp32 master of a plain step."""
    rng = np.random.default_rng(13)
    n = 4000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = [bf16_bits(rng.standard_normal(n) * 1e-3) for _ in range(6)]
    hp = dict(HP, lr=3.5e-6, weight_decay=0.01, wd_mode=1)
    ours, _, _ = run_oracle(orc, w0, grads, hp)
    w = w0.copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    mp = 1.0
    for t, g in enumerate(grads, start=1):
        k, mp = orc.nadam_scalars(t, hp["lr"], 0.9, 0.999, 1e-8, 0.01, True, True, 0.004, mp)
        orc.nadam_step_fp32(w, m, v, g, k)
    assert np.array_equal(ours.view(np.uint32), w.view(np.uint32))


def test_low_bits_accumulate_sub_bf16_updates(orc):
    """Updates far below one bf16 step still move the live bf16 weight through the residual."""
    n = 5000
    w0 = np.full(n, 1.0, np.float32)
    g = bf16_bits(np.full(n, 1e-3))
    hp = dict(HP, eps=0.0, nesterov=0, lr=2.0 ** -12)   # 1/32 of a bf16 step at 1.0
    t = make_tensor(orc, w0, small=False)
    st = orc.NadamState(1)
    for step in range(1, 65):
        orc.nadam_group_step([t], [g], st, step, hp)
    w = orc.kahan_merge(t["hi"], t["lo"])
    assert np.all(bits_to_f32(t["hi"]) < 1.0)          # the bf16 weight moved
    assert np.all(np.abs(w - (1.0 - 64 * 2.0 ** -12)) < 2e-3 * 64 * 2.0 ** -12)
    t2 = dict(hi=bf16_bits(w0), lo=None, m=np.full(n, 32768, np.uint16), v=np.zeros(n, np.uint16))
    st2 = orc.NadamState(1)
    for step in range(1, 65):
        orc.nadam_group_step([t2], [g], st2, step, hp)
    assert np.all(bits_to_f32(t2["hi"]) == 1.0)         # without the residual the update is lost


def test_zero_grad_and_decay_only(orc):
    rng = np.random.default_rng(14)
    for n in (2048, 10000):
        w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
        z = np.zeros(n, np.uint16)
        w, _, _ = run_oracle(orc, w0, [z] * 5, dict(HP), small=n <= 4096)
        assert np.array_equal(w, w0)
        lr, wd, T = 1e-2, 0.1, 7
        w, _, _ = run_oracle(orc, w0, [z] * T, dict(HP, lr=lr, weight_decay=wd, wd_mode=1), small=n <= 4096)
        expect = w0.astype(np.float64) * (1 - np.float64(np.float32(lr * wd))) ** T
        assert np.all(np.abs(w - expect) <= T * np.spacing(np.abs(w0)))


def test_u16_states_track_fp32_states(orc):
    """Above 4096 elements the moments are u16-companded; the trajectory stays within the codec's
    error of the fp32-moment trajectory (a loose property check, not an exact pin)."""
    rng = np.random.default_rng(15)
    n, steps = 8192, 10
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = [bf16_bits(rng.standard_normal(n) * 1e-3) for _ in range(steps)]
    hp = dict(HP, lr=1e-3)
    w_u16, t, st = run_oracle(orc, w0, grads, hp, small=False)
    ref = _torch_traj(torch.optim.NAdam, w0, grads, lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                      momentum_decay=0.004)
    d_u16 = w_u16.astype(np.float64) - w0
    d_ref = ref.astype(np.float64) - w0
    rel = np.abs(d_u16 - d_ref).sum() / np.abs(d_ref).sum()
    assert rel < 0.02
    s_m, s_v, a_m, a_v = st.scale(0)
    assert 0 < a_m <= s_m * 1.0001 and 0 < a_v <= s_v * 1.0001


def test_scale_is_a_bound(orc):
    """S_m(t) = b1 A_m(t-1) + (1-b1) G(t) bounds every |m(t)|, so codes rarely saturate."""
    rng = np.random.default_rng(16)
    n = 20000
    t = make_tensor(orc, (rng.standard_normal(n) * 0.02).astype(np.float32), small=False)
    st = orc.NadamState(1)
    for step in range(1, 6):
        g = bf16_bits(rng.standard_normal(n) * 1e-3 * step)
        orc.nadam_group_step([t], [g], st, step, dict(HP))
        s_m, s_v, a_m, a_v = st.scale(0)
        assert a_m <= s_m * (1 + 1e-4) and a_v <= s_v * (1 + 1e-4)
        sat = np.mean((t["m"] == 1) | (t["m"] == 65535))
        assert sat < 0.01


def test_f24_moments_are_truncated_fp32(orc):
    """f24 storage: each stored moment is the fp32 moment of a plain fp32-moment step truncated to
    its upper 24 bits, step after step (checked by replaying each step from the stored state)."""
    rng = np.random.default_rng(17)
    n = 10003
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    hi, lo = orc.kahan_split(w0)
    m = np.zeros(orc.f24_nbytes(n), np.uint8)
    v = np.zeros(orc.f24_nbytes(n), np.uint8)
    mp = 1.0
    for t in range(1, 6):
        g = bf16_bits(rng.standard_normal(n) * 1e-3)
        k, mp = orc.nadam_scalars(t, 1e-3, 0.9, 0.999, 1e-8, 0.0, False, True, 0.004, mp)
        # reference: the same step with fp32 moments started from the decoded f24 state
        w_ref = orc.kahan_merge(hi, lo).copy()
        m_ref = orc.f24_merge(m, n).copy()
        v_ref = orc.f24_merge(v, n).copy()
        orc.nadam_step_fp32(w_ref, m_ref, v_ref, g, k)
        orc.nadam_step_tensor_f24(hi, lo, m, v, g, k)
        assert np.array_equal(orc.kahan_merge(hi, lo).view(np.uint32), w_ref.view(np.uint32))
        mask = np.uint32(0xFFFFFF00)
        assert np.array_equal(orc.f24_merge(m, n).view(np.uint32), m_ref.view(np.uint32) & mask)
        assert np.array_equal(orc.f24_merge(v, n).view(np.uint32), v_ref.view(np.uint32) & mask)
    # 8 more mantissa bits than bf16: relative storage error below 2^-15
    x = (rng.standard_normal(1000) * 1e-4).astype(np.float32)
    rel = np.abs(orc.f24_merge(orc.f24_split(x), x.size) - x) / np.abs(x)
    assert rel.max() < 2.0 ** -15
    # storage layout: the padding between the two planes stays zero, the byte plane starts at 2n
    # rounded up to 16, and the upper plane holds the top 16 bits
    pad = slice(2 * n, orc.f24_lo_offset(n))
    assert orc.f24_lo_offset(n) == 20016 and pad.stop - pad.start == 10
    assert not m[pad].any() and not v[pad].any()
    y = np.array([1.0, -2.5, 3.0e-7], np.float32)
    buf = orc.f24_split(y)
    assert buf.size == 16 + 3
    assert list(buf[:6].view(np.uint16)) == [0x3F80, 0xC020, (y.view(np.uint32)[2] >> 16)]
    assert list(buf[16:]) == [0, 0, (y.view(np.uint32)[2] >> 8) & 0xFF]


def _scale_fixture(n=6000, seed=18):
    """Two hand-shaped gradients of a tensor above 4096 elements (u16 moments): random values of
    magnitude ~1e-3 plus one planted extreme, so that G = max|g| is a chosen power-of-two multiple
    (G1 = 2^-7 at t = 1, G2 = 3 * 2^-8 at t = 2)."""
    rng = np.random.default_rng(seed)
    g1 = rng.standard_normal(n) * 1e-3
    g1[17] = -2.0 ** -7
    g2 = rng.standard_normal(n) * 1e-3
    g2[4321] = 3.0 * 2.0 ** -8
    return bf16_bits(g1), bf16_bits(g2)


def _close(a, b, rel=4 * 2.0 ** -24):
    return abs(float(a) - float(b)) <= rel * abs(float(b))


@pytest.mark.parametrize("sr", [False, True])
def test_scale_record_closed_form(orc, sr):
    """The per-tensor scale record written out by hand (reading R4: the scale of step t bounds the
    moments of step t; sd-scripts PR #2187, second post, says only that the moments are
    scaled).  With b = beta and A(0) = 0:
        t = 1:  S_m = (1-b1) G1,  S_v = (1-b2) G1^2,  A_m = max|m1|, A_v = max v1 with
                m1 = (1-b1) g1 and v1 = (1-b2) g1^2 (fresh moments decode to 0 exactly);
        t = 2:  S_m = b1 A_m(1) + (1-b1) G2,  S_v = b2 A_v(1) + (1-b2) G2^2,
                A_m(2), A_v(2) the maxima of the step-2 moments, within the codec's error of the
                same moments computed in double from exact m1, v1.
    G enters S_v squared: S_v ~ 1e-3 * G^2 here, three orders of magnitude below (1-b2) G.
    Both store paths carry the record: the Kahan store and stochastic rounding (no residual).
    The hyper-parameters are fp32 values, so b is the fp32 number nearest 0.9 (0.999)."""
    b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))
    g1, g2 = _scale_fixture()
    n = g1.size
    G1, G2 = float(bits_to_f32(g1).__abs__().max()), float(bits_to_f32(g2).__abs__().max())
    assert G1 == 2.0 ** -7 and G2 == 3.0 * 2.0 ** -8
    w0 = (np.random.default_rng(19).standard_normal(n) * 0.02).astype(np.float32)
    t = make_tensor(orc, w0, small=False)
    st = orc.NadamState(1)
    mp = 1.0
    recs = []
    for step, g in enumerate((g1, g2), start=1):
        k, mp = orc.nadam_scalars(step, 1e-3, b1, b2, 1e-8, 0.0, False, True, 0.004, mp)
        if sr:
            orc.nadam_step_tensor_sr(t["hi"], t["m"], t["v"], g, st.scales[0], k, 7, 0, step)
        else:
            orc.nadam_step_tensor(t["hi"], t["lo"], t["m"], t["v"], g, st.scales[0], k)
        recs.append(st.scale(0))
    (s_m1, s_v1, a_m1, a_v1), (s_m2, s_v2, a_m2, a_v2) = recs
    # t = 1: closed forms in double
    assert _close(s_m1, (1 - b1) * G1), (s_m1, (1 - b1) * G1)
    assert _close(s_v1, (1 - b2) * G1 * G1), (s_v1, (1 - b2) * G1 * G1)
    x1 = bits_to_f32(g1).astype(np.float64)
    m1, v1 = (1 - b1) * x1, (1 - b2) * x1 * x1
    assert _close(a_m1, np.abs(m1).max()) and _close(a_v1, v1.max())
    # t = 2: the recurrence on the recorded maxima, in double
    assert _close(s_m2, b1 * a_m1 + (1 - b1) * G2, rel=8 * 2.0 ** -24)
    assert _close(s_v2, b2 * a_v1 + (1 - b2) * G2 * G2, rel=8 * 2.0 ** -24)
    x2 = bits_to_f32(g2).astype(np.float64)
    m2, v2 = b1 * m1 + (1 - b1) * x2, b2 * v1 + (1 - b2) * x2 * x2
    # decoded m1, v1 differ from the exact ones by at most half a code step in y: about
    # 2 * 0.5/32767 of S_m and 4 * 0.5/65535 of S_v (relative to the scale, not the value)
    assert abs(a_m2 - np.abs(m2).max()) <= b1 * s_m1 * 1.0 / 32767 + 1e-7 * a_m2
    assert abs(a_v2 - v2.max()) <= b2 * s_v1 * 2.0 / 65535 + 1e-7 * a_v2
    # both records bound what they describe
    assert a_m1 <= s_m1 * (1 + 2.0 ** -20) and a_v1 <= s_v1 * (1 + 2.0 ** -20)
    assert a_m2 <= s_m2 * (1 + 2.0 ** -20) and a_v2 <= s_v2 * (1 + 2.0 ** -20)
