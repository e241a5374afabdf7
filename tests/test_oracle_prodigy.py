"""Pins of the oracle's Prodigy mode and its step-size estimate d over the factored step: the
numerator factor d, the sampled-element layout, d under a constant gradient (where the update
clip is always active and the method reduces to a scalar recurrence), the independence of d
from the slicing when every sampled block looks alike, and d's monotonicity."""
import numpy as np

from test_oracle_nadam import bf16_bits

HP = dict(lr=1.0, beta2=0.99, decay_rate=-0.8, eps1=1e-30, eps2=0.0, clip_threshold=1.0, weight_decay=0.0)


def vector_tensor(orc, x0, slice_p):
    hi, lo = orc.kahan_split(np.asarray(x0, np.float32))
    p0, s = orc.prodigy_snapshot(hi, lo, slice_p)
    return dict(hi=hi, lo=lo, shape=(x0.size,), V=np.zeros(x0.size, np.float32), p0=p0, s=s)


def test_numerator_carries_d(orc):
    """Prodigy mode, t = 1, no clip, eps2 = 0: V = d^2 (1-b2) g^2, so u = d g / sqrt(V) =
    sign(g) / sqrt(1-b2) and the weight moves by d lr sign(g) / sqrt(1-b2).  Without the
    numerator d the move would be 1/d times larger."""
    rng = np.random.default_rng(60)
    n = 500
    g = bf16_bits(rng.standard_normal(n) * 1e-3)
    hi, lo = orc.kahan_split(np.zeros(n, np.float32))
    d, lr, b2 = 2.0 ** -10, 2.0 ** -4, 0.99
    k = orc.factored_scalars(1, lr, b2, -0.8, 0.0, 0.0, d, 1e30, 0.0, 1)
    V = np.zeros(n, np.float32)
    orc.factored_step_vector(hi, lo, g, V, k)
    w = orc.kahan_merge(hi, lo).astype(np.float64)
    gf = (g.astype(np.uint32) << 16).view(np.float32)
    expect = -d * lr * np.sign(gf) / np.sqrt(1.0 - b2)
    assert np.allclose(w, expect, rtol=1e-5, atol=0)


def test_snapshot_layout(orc):
    """n = 400, slice_p = 3: blocks 0, 3, 6 (elements 0-63, 192-255, 384-399) in order, 64
    entries per block, zero past the end; s starts at zero."""
    x = (np.arange(400, dtype=np.float32) + 1) * np.float32(0.25)
    hi, lo = orc.kahan_split(x)
    p0, s = orc.prodigy_snapshot(hi, lo, 3)
    assert orc.prodigy_slice_len(400, 3) == 192 and p0.size == 192
    assert np.array_equal(p0[:64], x[:64]) and np.array_equal(p0[64:128], x[192:256])
    assert np.array_equal(p0[128:144], x[384:400]) and not p0[144:].any() and not s.any()
    assert orc.prodigy_slice_len(0, 5) == 0 and orc.prodigy_slice_len(64, 1) == 64
    assert orc.prodigy_slice_len(65, 1) == 128 and orc.prodigy_slice_len(640, 11) == 64


def test_constant_gradient_recurrence(orc):
    """All n elements share g0 > 0, x0 = 0, eps2 = 0, clip 1.  Then V < d^2 g0^2, so u = d g0 /
    sqrt(V) > 1 and the clip makes every step move x by exactly lr d (fp32 d).  With D_k the
    displacement after k steps, the statistics reduce to dot = n g0 D_k and s = beta3 s + c g0
    (c = lr d^2): a scalar recurrence, computed here in float64."""
    n, g0, d0, b3, steps = 64, 2.0 ** -8, 1e-6, float(np.float32(np.sqrt(0.99))), 14
    hp = dict(HP)
    g = np.full(n, bf16_bits(np.array([g0]))[0], np.uint16)
    st = orc.ProdigyState(d0, b3, 1)
    t = vector_tensor(orc, np.zeros(n, np.float32), 1)
    # scalar recurrence
    d, r, s, D = d0, 0.0, 0.0, 0.0
    ds_ref, ds = [], []
    for k in range(1, steps + 1):
        df = float(np.float32(d))
        c = hp["lr"] * df * df
        cs = float(np.float32(c))
        s = b3 * s + cs * g0
        r = b3 * r + c * n * g0 * D
        D += hp["lr"] * df
        if s > 0 and r / (n * s) > d:
            d = r / (n * s)
        ds_ref.append(d)
        orc.prodigy_step(st, [([t], [g], hp)], k)
        ds.append(st.d.value)
    assert np.allclose(ds, ds_ref, rtol=1e-5, atol=0)
    assert ds[0] == d0 and ds[-1] > 100 * d0          # d starts at d0 and grows
    x = orc.kahan_merge(t["hi"], t["lo"]).astype(np.float64)
    assert np.allclose(x, -D, rtol=1e-5)


def test_d_independent_of_slicing_for_alike_blocks(orc):
    """When every 64-element block of a tensor holds the same values (weights and gradients),
    each sampled block contributes the same to both sums, so d does not depend on slice_p."""
    rng = np.random.default_rng(61)
    nb = 120                                 # 16-periodic values: 30 alike 64-element blocks
    x0 = np.tile((rng.standard_normal(16) * 0.02).astype(np.float32), nb)
    bias = rng.standard_normal(16) * 1e-3
    grads = [np.tile(bf16_bits(bias + rng.standard_normal(16) * 2e-4), nb) for _ in range(8)]
    runs = {}
    for P in (1, 7):
        st = orc.ProdigyState(1e-4, 0.995, P)
        t = vector_tensor(orc, x0, P)
        seq = []
        for k, g in enumerate(grads, start=1):
            orc.prodigy_step(st, [([t], [g], dict(HP, lr=0.5))], k)
            seq.append(st.d.value)
        runs[P] = (seq, orc.kahan_merge(t["hi"], t["lo"]).copy())
    assert np.allclose(runs[1][0], runs[7][0], rtol=1e-12, atol=0)
    assert runs[1][0][-1] > 1e-4
    assert np.array_equal(runs[1][1].view(np.uint32), runs[7][1].view(np.uint32))


def test_d_monotone_and_first_step(orc):
    """A matrix and a vector in two groups, random gradients with a persistent component: d
    after step 1 is d0 (x = p0, so the numerator is zero) and never decreases."""
    rng = np.random.default_rng(62)
    st = orc.ProdigyState(1e-5, 0.99, 3)
    shapes = [(40, 70), (333,)]
    groups = []
    for i, shp in enumerate(shapes):
        n = int(np.prod(shp))
        x0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
        t = vector_tensor(orc, x0, 3)
        t["shape"] = shp
        if len(shp) == 2:
            del t["V"]
            t["row"] = np.zeros(shp[0], np.float32)
            t["col"] = np.zeros(shp[1], np.float32)
        groups.append(([t], rng.standard_normal(n) * 1e-3, dict(HP, lr=0.3 + 0.2 * i)))
    seq = []
    for k in range(1, 11):
        step = [([t], [bf16_bits(base + rng.standard_normal(base.size) * 5e-4)], hp) for ([t], base, hp) in groups]
        orc.prodigy_step(st, step, k)
        seq.append(st.d.value)
    assert seq[0] == 1e-5
    assert all(b >= a for a, b in zip(seq, seq[1:]))
    assert seq[-1] > seq[0]
