"""Pins of the oracle's Adan step (Algorithm 1 of the Adan paper the pages link, fp32 states):
closed forms for constant and two-valued gradient sequences, and the decay factor."""
import numpy as np

from test_oracle_nadam import bf16_bits, bits_to_f32

B1, B2, B3 = 0.02, 0.08, 0.01


def run(orc, w0, grads, lr, wd=0.0, eps=0.0):
    n = w0.size
    hi, lo = orc.kahan_split(w0)
    mnv = np.zeros(3 * orc.adan_plane(n), np.float32)
    gp = np.zeros(n, np.uint16)
    k = orc.adan_scalars(lr, B1, B2, B3, eps, wd)
    for t, g in enumerate(grads, start=1):
        orc.adan_step_tensor(hi, lo, mnv, gp, g, t, k)
    return orc.kahan_merge(hi, lo).astype(np.float64), mnv, gp


def test_constant_gradient_moves_by_lr_sign():
    """Constant g: the difference is zero, so v = 0, m = g, n = g^2 at every step and each step
    is exactly w - lr sign(g) (eps = 0, no decay)."""
    import oracle as orc
    rng = np.random.default_rng(40)
    n = 2003
    g = bf16_bits(rng.choice([-1.0, 1.0], n) * 2.0 ** rng.integers(-12, -4, n))
    lr = 2.0 ** -10
    w, mnv, gp = run(orc, np.zeros(n, np.float32), [g] * 6, lr)
    assert np.array_equal(w, -6 * lr * np.sign(bits_to_f32(g)))
    # planes at 0, P, 2P with P = n rounded up to 4; the padding stays zero
    P = orc.adan_plane(n)
    assert P == 2004 and mnv.size == 3 * P
    gf = bits_to_f32(g)
    assert np.array_equal(mnv[:n], gf) and np.all(mnv[P:P + n] == 0)
    assert np.array_equal(mnv[2 * P:2 * P + n], gf * gf)
    assert np.all(mnv[n:P] == 0) and np.all(mnv[2 * P + n:] == 0)
    assert np.array_equal(gp, g)


def test_two_gradients_closed_form():
    """g1 then g2: step 1 moves by -lr sign(g1); step 2 uses m = (1-b1) g1 + b1 g2, v = g2 - g1,
    n = (1-b3) g1^2 + b3 (g2 + (1-b2)(g2 - g1))^2 (computed here in float64)."""
    import oracle as orc
    rng = np.random.default_rng(41)
    n = 3000
    g1 = bf16_bits(rng.standard_normal(n) * 1e-3)
    g2 = bf16_bits(rng.standard_normal(n) * 1e-3)
    a, b = bits_to_f32(g1).astype(np.float64), bits_to_f32(g2).astype(np.float64)
    lr, eps = 1e-3, 1e-8
    w, _, _ = run(orc, np.zeros(n, np.float32), [g1, g2], lr, eps=eps)
    w1 = -lr * a / (np.abs(a) + eps)
    m = (1 - B1) * a + B1 * b
    v = b - a
    nn = (1 - B3) * a * a + B3 * (b + (1 - B2) * (b - a)) ** 2
    expect = w1 - lr * (m + (1 - B2) * v) / (np.sqrt(nn) + eps)
    # two steps of size ~lr each: fp32 rounding of each is a few ulps of lr (the sum may cancel)
    assert np.all(np.abs(w - expect) <= 2e-6 * lr)


def test_decay_only():
    import oracle as orc
    rng = np.random.default_rng(42)
    n = 1000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    z = np.zeros(n, np.uint16)
    lr, wd = 1e-2, 0.1
    w, _, _ = run(orc, w0, [z] * 5, lr, wd=wd, eps=1e-8)
    expect = w0.astype(np.float64) / (1 + lr * wd) ** 5
    assert np.all(np.abs(w - expect) <= 5 * np.spacing(np.abs(w0)))


def run_f24(orc, w0, grads, lr, wd=0.0, eps=0.0):
    n = w0.size
    hi, lo = orc.kahan_split(w0)
    buf = np.zeros(orc.adan_f24_nbytes(n), np.uint8)
    gp = np.zeros(n, np.uint16)
    k = orc.adan_scalars(lr, B1, B2, B3, eps, wd)
    for t, g in enumerate(grads, start=1):
        orc.adan_step_tensor_f24(hi, lo, buf, gp, g, t, k)
    return orc.kahan_merge(hi, lo).astype(np.float64), buf, gp


def test_f24_constant_gradient_closed_form_and_layout():
    """f24 states (above 4096 elements), constant gradient: m = g and n = g^2 have at most 16
    significant bits (g is bf16), so f24 stores them exactly and every step is w - lr sign(g), as
    with fp32 states.  Layout by hand for n = 5000: each state buffer holds 10000 bytes of upper
    words, then 5000 bytes of bits 8..15, padded to 15008; m at byte 0, v at 15008, n at 30016."""
    import oracle as orc
    rng = np.random.default_rng(43)
    n = 5000
    g = bf16_bits(rng.choice([-1.0, 1.0], n) * 2.0 ** rng.integers(-12, -4, n))
    lr = 2.0 ** -10
    w, buf, gp = run_f24(orc, np.zeros(n, np.float32), [g] * 4, lr)
    assert np.array_equal(w, -4 * lr * np.sign(bits_to_f32(g)))
    F = orc.adan_f24_stride(n)
    assert F == 15008 and buf.size == 3 * F == orc.adan_f24_nbytes(n)
    gb = bits_to_f32(g).view(np.uint32)
    g2 = (bits_to_f32(g) * bits_to_f32(g)).view(np.uint32)
    for j, want in ((0, gb), (1, np.zeros(n, np.uint32)), (2, g2)):
        sub = buf[j * F:(j + 1) * F]
        assert np.array_equal(sub[:2 * n].view(np.uint16), (want >> 16).astype(np.uint16))
        assert np.array_equal(sub[10000:15000], ((want >> 8) & 0xFF).astype(np.uint8))
        assert not sub[15000:].any()
    assert np.array_equal(gp, g)


def test_f24_states_are_truncated_fp32_states():
    """Replay: each step of the f24 path equals the fp32-state step started from the decoded f24
    states, with m, v, n stored truncated to their upper 24 bits and the Kahan weight bit-identical;
    4096 or fewer elements keep the fp32 planes (same results as the fp32 path)."""
    import oracle as orc
    rng = np.random.default_rng(44)
    lr, eps, wd = 1e-3, 1e-8, 0.02
    k = orc.adan_scalars(lr, B1, B2, B3, eps, wd)
    for n in (4096, 10003):
        w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
        hi, lo = orc.kahan_split(w0)
        buf = np.zeros(orc.adan_f24_nbytes(n), np.uint8)
        gp = np.zeros(n, np.uint16)
        F = orc.adan_f24_stride(n)
        P = orc.adan_plane(n)
        mask = np.uint32(0xFFFFFF00)
        for t in range(1, 6):
            g = bf16_bits(rng.standard_normal(n) * 1e-3)
            hi_r, lo_r, gp_r = hi.copy(), lo.copy(), gp.copy()
            if n > 4096:
                mnv = np.zeros(3 * P, np.float32)
                for j in range(3):
                    mnv[j * P:j * P + n] = orc.f24_merge(buf[j * F:j * F + orc.f24_nbytes(n)], n)
            else:
                mnv = buf.view(np.float32).copy()
            orc.adan_step_tensor(hi_r, lo_r, mnv, gp_r, g, t, k)
            orc.adan_step_tensor_f24(hi, lo, buf, gp, g, t, k)
            assert np.array_equal(hi, hi_r) and np.array_equal(lo, lo_r) and np.array_equal(gp, gp_r)
            if n > 4096:
                for j in range(3):
                    got = orc.f24_merge(buf[j * F:j * F + orc.f24_nbytes(n)], n).view(np.uint32)
                    assert np.array_equal(got, mnv[j * P:j * P + n].view(np.uint32) & mask), (t, j)
            else:
                assert np.array_equal(buf.view(np.float32), mnv)
