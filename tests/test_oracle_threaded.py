"""The oracle's threaded timing driver (the same oracle.c built with OpenMP) against the
single-threaded oracle: bit-identical weights, residuals, codes, fp32 moments and scale records
over several steps, for tensors cut into many slices, small tensors and tensors without a
residual.  This is what lets the benchmark time the oracle on every host core."""
import numpy as np

from test_oracle_nadam import HP, bf16_bits, make_tensor


def test_threaded_driver_is_bit_identical(orc):
    rng = np.random.default_rng(70)
    sizes = [3_000_001, 1 << 20, 4096, 4097, 77, 2_500_000, 150_000]
    hp = dict(HP, weight_decay=0.01, wd_mode=1)
    a, b = [], []
    for i, n in enumerate(sizes):
        w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
        t1, t2 = make_tensor(orc, w0, n <= 4096), make_tensor(orc, w0, n <= 4096)
        if i == 5:                         # no residual: round-to-nearest store
            t1["lo"] = t2["lo"] = None
        a.append(t1)
        b.append(t2)
    sa, sb = orc.NadamState(len(sizes)), orc.NadamState(len(sizes))
    for step in range(1, 4):
        grads = [bf16_bits(rng.standard_normal(n) * 1e-3 * step) for n in sizes]
        grads[0][123_456] = 0                 # exact zeros and a planted maximum in a late slice
        grads[0][2_900_000] = bf16_bits(np.array([0.05]))[0]
        orc.nadam_group_step(a, grads, sa, step, hp)
        orc.nadam_group_step_mt(b, grads, sb, step, hp)
        for i, (x, y) in enumerate(zip(a, b)):
            for key in ("hi", "lo", "m", "v"):
                if x[key] is None:
                    continue
                assert np.array_equal(x[key].view(np.uint8), y[key].view(np.uint8)), (step, i, key)
            assert np.array_equal(np.float32(sa.scale(i)), np.float32(sb.scale(i))), (step, i)
    assert sa.mu_product.value == sb.mu_product.value
    assert orc.threads() >= 1
