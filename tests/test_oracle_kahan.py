"""Pins of the oracle's Kahan split/merge and bf16 store.

The residual is the 16 low bits clipped from the f32 value and the live weight is its bf16 upper
half, so that the bit-identical f32 value is restored ("Kahan summation for Adafactor-optimized
Flux FFT", sd-scripts PR #2159, first comment; bf16 as the high half of an f32 pattern,
"Amazing Flux FFT quality on a 5090", sd-scripts PR #2187, third post).
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixtures():
    rows = []
    with open(os.path.join(GOLDEN, "kahan_ieee_bits.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            dec, bits, hi, lo = line.split()
            rows.append((dec, int(bits, 16), int(hi, 16), int(lo, 16)))
    return rows


def test_ieee_fixtures(orc):
    rows = _fixtures()
    x = np.array([np.float32(float(d)) for d, _, _, _ in rows], dtype=np.float32)
    # the fixture's pattern is the IEEE encoding of the decimal (numpy's parser is independent)
    assert [int(b) for b in x.view(np.uint32)] == [b for _, b, _, _ in rows]
    hi, lo = orc.kahan_split(x)
    assert [int(h) for h in hi] == [h for _, _, h, _ in rows]
    assert [int(v) for v in lo] == [v for _, _, _, v in rows]
    back = orc.kahan_merge(hi, lo)
    assert np.array_equal(back.view(np.uint32), x.view(np.uint32))


@pytest.mark.slow
def test_split_merge_exhaustive(orc):
    """merge(split(x)) is the identity on all 2^32 patterns, NaN payloads and -0 included.  The
    buffers are reused chunk after chunk (allocation, not arithmetic, dominated this test)."""
    chunk = 1 << 24
    base = np.arange(chunk, dtype=np.uint32)
    bits = np.empty(chunk, np.uint32)
    hi, lo = np.empty(chunk, np.uint16), np.empty(chunk, np.uint16)
    back = np.empty(chunk, np.float32)
    halves = bits.view(np.uint16)          # little-endian: [2i] the low half, [2i + 1] the high half
    assert np.little_endian
    for start in range(0, 1 << 32, chunk):
        np.add(base, np.uint32(start), out=bits)
        orc.kahan_split(bits.view(np.float32), hi, lo)
        # the halves are the upper and lower 16 bits of the pattern
        assert np.array_equal(hi, halves[1::2])
        assert np.array_equal(lo, halves[0::2])
        orc.kahan_merge(hi, lo, back)
        assert np.array_equal(back.view(np.uint32), bits)


def test_hi_is_truncation_toward_zero(orc):
    """The live bf16 weight never exceeds |x| and is within one bf16 step of it."""
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200_000) * rng.choice([1e-30, 1e-3, 1.0, 1e20], 200_000)).astype(np.float32)
    hi, _ = orc.kahan_split(x)
    h = torch.from_numpy(hi.astype(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    xd = x.astype(np.float64)
    assert np.all(np.abs(h) <= np.abs(xd))
    assert np.all(np.sign(h) * np.sign(xd) >= 0)
    step = np.abs(h) * 2.0 ** -7 + 1e-300
    assert np.all(np.abs(xd - h) < step * 1.0000001 + np.abs(xd) * 2.0 ** -7)


def test_round_bf16_matches_torch(orc):
    """The no-residual store is IEEE round-to-nearest-even, as torch's bf16 cast."""
    rng = np.random.default_rng(2)
    upper = rng.integers(0, 1 << 16, 300_000, dtype=np.uint32)
    lower = rng.choice(np.array([0x0000, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234], np.uint32), 300_000)
    bits = (upper << 16) | lower
    x = bits.view(np.float32)
    finite = np.isfinite(x)
    ours = orc.round_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(ours[finite], ref[finite])
    nan = np.isnan(x)
    back = torch.from_numpy(ours[nan].astype(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.all(np.isnan(back))
