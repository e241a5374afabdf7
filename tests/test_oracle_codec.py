"""Pins of the oracle's companded u16 state codec.

The pages fix the scheme -- per-tensor scaling, a biased uint16, a pow() curve spreading the
roughly exponential values over 0..65535 -- but not its constants ("Amazing Flux FFT quality on
a 5090", sd-scripts PR #2187, second post).  The build fixes exponent 1/2 with bias 32768 for
exp_avg and exponent 1/4 without bias for exp_avg_sq; these tests pin the oracle to that
definition by hand-worked codes, exhaustive round trips, the half-step bound and monotonicity.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALES = [1e-12, 3.7e-5, 1.0, 123.4, 2.0 ** 20]


def test_hand_worked_codes(orc):
    with open(os.path.join(GOLDEN, "codec_fixtures.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 20
    for kind, s, x, code in rows:
        s, x, code = np.float32(s), np.float32(x), int(code)
        c = orc.codec_consts(float(s), float(s))
        if kind == "m":
            got = orc.encode_m(float(x), c.rm)
        else:
            got = orc.encode_v(float(np.sqrt(np.float32(x))), c.rv)
        assert got == code, (kind, s, x, got, code)


@pytest.mark.parametrize("s", SCALES)
def test_roundtrip_every_code(orc, s):
    """encode(decode(c)) == c for all 65535 exp_avg codes and all 65536 exp_avg_sq codes."""
    s = float(np.float32(s))
    k = orc.codec_consts(s, s)
    codes = np.arange(65536, dtype=np.uint16)
    mdec = orc.state_unpack(codes, s, True)
    vdec = orc.state_unpack(codes, s, False)
    for c in range(1, 65536):
        assert orc.encode_m(float(mdec[c]), k.rm) == c
    for c in range(65536):
        assert orc.encode_v(float(np.sqrt(vdec[c])), k.rv) == c
    # the decoded end points are the scale itself (to a few ulps) and zero
    assert abs(mdec[65535] - s) <= 4 * np.spacing(np.float32(s)) and mdec[32768] == 0.0
    assert abs(vdec[65535] - s) <= 8 * np.spacing(np.float32(s)) and vdec[0] == 0.0


def test_half_step_bound_and_monotone(orc):
    rng = np.random.default_rng(3)
    s = np.float32(2.5e-4)
    x = np.sort((rng.uniform(-1, 1, 20000) * s).astype(np.float32))
    x = np.clip(x, -s, s)
    codes, _ = orc.state_pack(np.append(x, s).astype(np.float32), True)
    codes = codes[:-1]
    dec = orc.state_unpack(codes, float(s), True).astype(np.float64)
    y_true = np.sqrt(np.abs(x.astype(np.float64)) / float(s))
    y_dec = np.sqrt(np.abs(dec) / float(s))
    assert np.max(np.abs(y_true - y_dec)) <= (0.5 + 0.02) / 32767   # half a code plus a few fp32 ulps of y
    assert np.all(np.diff(codes.astype(np.int64)) >= 0)          # monotone in x
    assert np.all(np.sign(dec) * np.sign(x) >= 0)

    v = np.sort((rng.uniform(0, 1, 20000) ** 6 * s).astype(np.float32))
    vcodes, vs = orc.state_pack(np.append(v, s).astype(np.float32), False)
    assert vs == s
    vcodes = vcodes[:-1]
    vdec = orc.state_unpack(vcodes, float(s), False).astype(np.float64)
    z_true = (v.astype(np.float64) / float(s)) ** 0.25
    z_dec = (vdec / float(s)) ** 0.25
    assert np.max(np.abs(z_true - z_dec)) <= (0.5 + 0.02) / 65535
    assert np.all(np.diff(vcodes.astype(np.int64)) >= 0)


def test_pack_scale_is_absmax(orc):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(5000) * 1e-3).astype(np.float32)
    codes, s = orc.state_pack(x, True)
    assert s == np.max(np.abs(x))
    assert codes[np.argmax(np.abs(x))] in (1, 65535)
    z = np.zeros(100, np.float32)
    codes, s = orc.state_pack(z, True)
    assert s == 0.0 and np.all(codes == 32768)
    codes, s = orc.state_pack(z, False)
    assert s == 0.0 and np.all(codes == 0)
    assert np.all(orc.state_unpack(codes, 0.0, False) == 0)


def test_codec_error_vs_bf16(orc):
    """Reports the codec's L1 error against a bf16 cast on moment-like data (the pages quote a
    ~90% reduction for their scheme; this only asserts the u16 codec is the better of the two)."""
    import torch
    rng = np.random.default_rng(5)
    g = rng.standard_normal(1 << 16) * 1e-4
    m = (0.1 * g).astype(np.float32)
    v = (0.001 * g * g).astype(np.float32)
    for x, signed in ((m, True), (v, False)):
        codes, s = orc.state_pack(x, signed)
        dec = orc.state_unpack(codes, s, signed)
        bf = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
        e_u16 = np.abs(dec.astype(np.float64) - x).sum()
        e_bf = np.abs(bf.astype(np.float64) - x).sum()
        assert e_u16 < e_bf
