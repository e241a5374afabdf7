"""Pins of the oracle's stochastic rounding: its Philox4x32-10 against the generator's published
known-answer vectors, the element-to-lane layout, exactness on bf16 values, and the rounding
probability equal to the distance to the lower bf16 neighbour."""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_philox_known_answers(orc):
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        w = [int(x, 16) for x in r]
        assert list(orc.philox4x32_10(w[0:4], w[4:6])) == w[6:10]


def test_sr_lanes_cover_the_block(orc):
    """Eight consecutive elements from i = 8b take the eight 16-bit halves of one block, low half
    first; the block's counter is (b, tensor, step) under key seed, and blocks differ."""
    seed, tensor, step = 0x1234567890ABCDEF, 7, 3
    b = (1 << 33) + 5                      # a block index above 2^32: both counter words used
    out = orc.philox4x32_10([b & 0xFFFFFFFF, b >> 32, tensor, step], [seed & 0xFFFFFFFF, seed >> 32])
    lanes = [orc.sr_bits(seed, tensor, step, 8 * b + j) for j in range(8)]
    assert lanes == [(int(out[j // 2]) >> (16 * (j % 2))) & 0xFFFF for j in range(8)]
    nxt = [orc.sr_bits(seed, tensor, step, 8 * (b + 1) + j) for j in range(8)]
    other_t = [orc.sr_bits(seed, tensor + 1, step, 8 * b + j) for j in range(8)]
    other_s = [orc.sr_bits(seed, tensor, step + 1, 8 * b + j) for j in range(8)]
    assert lanes != nxt and lanes != other_t and lanes != other_s


def test_sr_bits_uniform(orc):
    """The 16-bit lanes are uniform: chi-square over 64 bins of 65,536 draws (63 degrees of
    freedom; the 1e-6 tail is near 130)."""
    draws = np.array([orc.sr_bits(99, 1, 2, i) for i in range(65536)], np.uint32)
    counts = np.bincount(draws >> 10, minlength=64)
    e = draws.size / 64
    assert ((counts - e) ** 2 / e).sum() < 130


def test_sr_exact_on_bf16_values_and_keeps_specials(orc):
    x = torch.randn(10000).to(torch.bfloat16).float().numpy()
    out = orc.stochastic_round(x, 123, 0, 1)
    assert np.array_equal(out, (x.view(np.uint32) >> 16).astype(np.uint16))
    sp = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0], np.float32)
    back = (orc.stochastic_round(sp, 1, 2, 3).astype(np.uint32) << 16).view(np.float32)
    assert np.isposinf(back[0]) and np.isneginf(back[1]) and np.isnan(back[2]) and back[3] == 0 and back[4] == 0


@pytest.mark.parametrize("frac", [0.1, 0.5, 0.9])
def test_sr_probability_is_distance(orc, frac):
    """x = lower + frac * (upper - lower): over many independent draws the result is upper with
    probability frac, so the mean equals x (unbiased), within a 5-sigma binomial bound."""
    n = 200_000
    lower = np.float32(1.0)
    step = np.float32(2.0 ** -7)            # bf16 spacing in [1, 2)
    x = np.full(n, lower + np.float32(frac) * step, np.float32)
    out = orc.stochastic_round(x, 99, 5, 7)
    up = (out.astype(np.uint32) << 16).view(np.float32) > lower
    p = up.mean()
    assert abs(p - frac) < 5 * np.sqrt(frac * (1 - frac) / n)
    mean = ((out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)).mean()
    assert abs(mean - float(x[0])) < 5 * float(step) * np.sqrt(frac * (1 - frac) / n)


def test_sr_step_is_rounded_no_residual_step(orc):
    """The SR step equals the no-residual step's fp32 result stochastically rounded: replay with
    fp32 moments (n <= 4096) from the same state."""
    rng = np.random.default_rng(31)
    n = 3000
    w = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)).to(torch.bfloat16)
    hi = w.view(torch.int16).numpy().view(np.uint16).copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    st = orc.NadamState(1)
    mp = 1.0
    for t in range(1, 4):
        g = torch.from_numpy((rng.standard_normal(n) * 1e-3).astype(np.float32)).to(torch.bfloat16)
        gb = g.view(torch.int16).numpy().view(np.uint16)
        k, mp = orc.nadam_scalars(t, 1e-3, 0.9, 0.999, 1e-8, 0.0, False, True, 0.004, mp)
        w32 = (hi.astype(np.uint32) << 16).view(np.float32).copy()
        m2, v2 = m.copy(), v.copy()
        orc.nadam_step_fp32(w32, m2, v2, gb, k)
        expect = orc.stochastic_round(w32, 42, 3, t)
        orc.nadam_step_tensor_sr(hi, m, v, gb, st.scales[0], k, 42, 3, t)
        assert np.array_equal(hi, expect)
        assert np.array_equal(m.view(np.uint32), m2.view(np.uint32))
