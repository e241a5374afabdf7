"""GPU parity of the fused multi-tensor NAdam(W)/Adam + Kahan + u16-moment step against the oracle,
through the C ABI.  Weights, residuals and moment codes must be bit-identical to the oracle's
after every step; per-tensor scale records equal."""
import numpy as np
import pytest
import torch

from helpers import OracleNadam, alloc_offset, assert_nadam_equal, cuda_bits
from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(W.NADAM_HP)


@pytest.fixture(scope="module")
def eng():
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    return engine


def run_parity(orc, eng, shapes, steps, hp, seed=0, g_std=1e-3, zero_frac=0.0, kahan=True, check_every=True):
    masters = [W.master_weights(s, seed, i) for i, s in enumerate(shapes)]
    ora = OracleNadam(orc, [m.numpy() for m in masters], kahan=kahan)
    if kahan:
        grp = eng.NadamGroup.from_masters([m.cuda() for m in masters])
    else:
        grp = eng.NadamGroup([m.cuda().to(torch.bfloat16) for m in masters], kahan=False)
    for t in range(1, steps + 1):
        grads = [W.grad_bf16(s, seed, i, t, g_std, zero_frac=zero_frac) for i, s in enumerate(shapes)]
        ora.step([W.bits16(g).reshape(-1) for g in grads], hp)
        grp.step([g.cuda() for g in grads], hp)
        if check_every or t == steps:
            torch.cuda.synchronize()
            assert_nadam_equal(ora, grp, f"step {t}")
            got = grp.scales()
            for i, (a, b) in enumerate(zip(got, ora.scales())):
                if W.numel(shapes[i]) > 4096:
                    assert a == pytest.approx(b, rel=0, abs=0), (i, a, b)
    return ora, grp


@pytest.mark.parametrize("states", ["u16", "f24"])
def test_empty_tensors_in_a_group(orc, eng, states):
    """Tensors without elements (no gradient, nothing to update) among ordinary ones: the others
    step bit-identically to the oracle and the empty ones are left alone."""
    shapes = [(5000,), (0,), (3, 0), (300,), (0, 7), (20000,)]
    seed, hp = 12, dict(HP, lr=1e-3)
    masters = [W.master_weights(s, seed, i) for i, s in enumerate(shapes)]
    ora = OracleNadam(orc, [m.numpy() for m in masters])
    grp = eng.NadamGroup.from_masters([m.cuda() for m in masters], states=states)
    for t in range(1, 4):
        grads = [W.grad_bf16(s, seed, i, t, 1e-3) for i, s in enumerate(shapes)]
        if states == "u16":
            ora.step([W.bits16(g).reshape(-1) for g in grads], hp)
        grp.step([g.cuda() for g in grads], hp)
    torch.cuda.synchronize()
    from memory_lean_optimizer_gb300 import lmopt
    assert lmopt.optim_query_nonfinite(grp.handle) == 0
    assert all(grp.weights[i].numel() == 0 for i, s in enumerate(shapes) if W.numel(s) == 0)
    if states == "u16":
        assert_nadam_equal(ora, grp, "empty tensors")


def test_one_1024x1024_ten_steps(orc, eng):
    """The 1024x1024 single-tensor workload, NAdam, lr 3.5e-6, 10 steps, seed 0 (one launch per
    step: its chunks fit on the GPU at once)."""
    _, grp = run_parity(orc, eng, [(1024, 1024)], 10, HP, g_std=1e-3)
    assert grp.launches(HP) == 1


@pytest.mark.parametrize("sr", [False, True])
def test_one_launch_step_equals_two_launches(orc, eng, sr):
    """The one-launch step (pre-pass, grid barrier, update in one cooperative kernel) and the
    two-kernel step (optim_step_nadam_begin / _end) give the same bits, 1% exact-zero gradients
    included; a group too large for one launch reports two, and both agree with the oracle."""
    from memory_lean_optimizer_gb300 import lmopt
    shapes = [(4097,), (70001,), (300,), (2048, 96)]
    hp = dict(HP, lr=1e-3, stochastic_rounding=int(sr), seed=99)
    seed = 21
    masters = [W.master_weights(s, seed, i).cuda() for i, s in enumerate(shapes)]
    mk = (lambda: eng.NadamGroup([m.to(torch.bfloat16) for m in masters], kahan=False)) if sr else \
         (lambda: eng.NadamGroup.from_masters([m.clone() for m in masters]))
    one, two = mk(), mk()
    assert one.launches(hp) == 1
    for t in range(1, 4):
        grads = [W.grad_bf16(s, seed, i, t, 1e-3, zero_frac=0.01).cuda() for i, s in enumerate(shapes)]
        one.step(grads, hp)
        two.step_begin(grads, hp)
        two.step_end()
    torch.cuda.synchronize()
    for a, b in zip(one.weights + one.m + one.v, two.weights + two.m + two.v):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    if not sr:
        assert all(torch.equal(a, b) for a, b in zip(one.res, two.res))
    assert one.scales() == two.scales()
    assert lmopt.optim_query_nonfinite(one.handle) == 0
    big = eng.NadamGroup.from_masters([torch.zeros(40 * 16384 * 152, device="cuda")])
    assert big.launches(hp) == 2
    for g in (one, two, big):
        g.close()


@pytest.mark.parametrize("variant", ["adam", "nadam", "nadamw", "adamw"])
def test_ragged_group_all_paths(orc, eng, variant):
    """Sizes around every boundary: fp32-state (<=4096) and u16 tensors, ragged tails, several
    chunks, sizes not multiple of 8."""
    sizes = [1, 7, 8, 63, 64, 4095, 4096, 4097, 16383, 16384, 16385, 50001, 131075, 1 << 18]
    hp = dict(HP, lr=1e-4, nesterov=variant.startswith("n"),
              weight_decay=0.05 if variant.endswith("w") else 0.0, wd_mode=1 if variant.endswith("w") else 0)
    run_parity(orc, eng, [(n,) for n in sizes], 4, hp, seed=3, zero_frac=0.01)


def test_no_residual_store(orc, eng):
    """res = NULL: the weight is stored round-to-nearest-even, as the oracle's bf16 store."""
    sizes = [100, 5000, 40000]
    run_parity(orc, eng, [(n,) for n in sizes], 3, dict(HP, lr=1e-3), seed=4, kahan=False)


def test_misaligned_buffers_take_scalar_path(orc, eng):
    """Buffers 2-byte (not 16-byte) aligned go element by element and give identical bits."""
    from memory_lean_optimizer_gb300 import lmopt
    sizes = [3000, 20001, 70000]
    seed = 5
    masters = [W.master_weights((n,), seed, i) for i, n in enumerate(sizes)]
    ora = OracleNadam(orc, [m.numpy() for m in masters])
    keep, descs, ws, rs, ms, vs = [], [], [], [], [], []
    for i, n in enumerate(sizes):
        hi, lo = orc.kahan_split(masters[i].numpy())
        b1, w = alloc_offset(n, torch.int16, 1)
        b2, r = alloc_offset(n, torch.int16, 3)
        w.copy_(torch.from_numpy(hi.view(np.int16)))
        r.copy_(torch.from_numpy(lo.view(np.int16)))
        if n <= 4096:
            b3, m = alloc_offset(n, torch.float32, 1)
            b4, v = alloc_offset(n, torch.float32, 1)
        else:
            b3, m = alloc_offset(n, torch.int16, 5, fill=-32768)
            b4, v = alloc_offset(n, torch.int16, 7)
        keep += [b1, b2, b3, b4]
        d = lmopt.TensorDesc(w_bf16=w.data_ptr(), res_u16=r.data_ptr(), m=m.data_ptr(), v=v.data_ptr(),
                             numel=n, ndim=1)
        d.shape[0] = n
        descs.append(d)
        ws.append(w), rs.append(r), ms.append(m), vs.append(v)
    h = lmopt.optim_group_create(descs, lmopt.OPTIM_KIND_NADAM)
    hp = dict(HP, lr=1e-3)
    H = lmopt.NadamHparams(lr=hp["lr"], beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, wd_mode=0,
                           nesterov=1, momentum_decay=0.004)
    try:
        for t in range(1, 4):
            grads = [W.grad_bf16((n,), seed, i, t, 1e-3) for i, n in enumerate(sizes)]
            ora.step([W.bits16(g) for g in grads], hp)
            gbufs = []
            for g in grads:
                b, gg = alloc_offset(g.numel(), torch.int16, 1)
                gg.copy_(g.view(torch.int16))
                gbufs += [b, gg]
            lmopt.optim_step_nadam_kahan(h, [gbufs[2 * i + 1].data_ptr() for i in range(len(sizes))], t, H, 0)
            torch.cuda.synchronize()
            for i, ot in enumerate(ora.t):
                assert np.array_equal(cuda_bits(ws[i]), ot["hi"])
                assert np.array_equal(cuda_bits(rs[i]), ot["lo"])
                if sizes[i] > 4096:
                    assert np.array_equal(cuda_bits(ms[i]), ot["m"])
                    assert np.array_equal(cuda_bits(vs[i]), ot["v"])
                else:
                    assert np.array_equal(ms[i].cpu().numpy(), ot["m"])
    finally:
        lmopt.optim_group_destroy(h)


def test_ragged_log_uniform_small(orc, eng):
    """A reduced ragged workload: 400 tensors, sizes round(2^U(6,18)), 1% exact-zero grads."""
    sizes = W.ragged_sizes(400, seed=1, hi_exp=18.0)
    run_parity(orc, eng, [(n,) for n in sizes], 3, HP, seed=1, zero_frac=0.01, check_every=False)


def test_checkpoint_resume_bit_identical(orc, eng):
    """k steps, save (codes, residuals, scales, step, mu product), restore into a new group,
    N-k more steps == N uninterrupted steps."""
    from memory_lean_optimizer_gb300 import lmopt
    shapes = [(5000,), (70000,), (300,)]
    seed = 6
    masters = [W.master_weights(s, seed, i) for i, s in enumerate(shapes)]
    grads = {t: [W.grad_bf16(s, seed, i, t, 1e-3) for i, s in enumerate(shapes)] for t in range(1, 6)}
    a = eng.NadamGroup.from_masters([m.cuda() for m in masters])
    for t in range(1, 6):
        a.step([g.cuda() for g in grads[t]], HP)
    b = eng.NadamGroup.from_masters([m.cuda() for m in masters])
    for t in range(1, 4):
        b.step([g.cuda() for g in grads[t]], HP)
    recs = b.scales()
    step, mp = lmopt.optim_group_get_step(b.handle)
    c = eng.NadamGroup([w.clone() for w in b.weights], [r.clone() for r in b.res])
    for i in range(len(shapes)):
        c.m[i].copy_(b.m[i])
        c.v[i].copy_(b.v[i])
    lmopt.optim_set_scales(c.handle, recs)
    lmopt.optim_group_set_step(c.handle, step, mp)
    c.step_count = step
    for t in range(4, 6):
        c.step([g.cuda() for g in grads[t]], HP)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        assert torch.equal(a.weights[i].view(torch.int16), c.weights[i].view(torch.int16))
        assert torch.equal(a.res[i], c.res[i])
        assert torch.equal(a.m[i].view(torch.int32) if a.m[i].dtype == torch.float32 else a.m[i],
                           c.m[i].view(torch.int32) if c.m[i].dtype == torch.float32 else c.m[i])


def test_nonfinite_counter_and_step_validation(eng):
    from memory_lean_optimizer_gb300 import lmopt
    n = 10000
    grp = eng.NadamGroup.from_masters([torch.randn(n, device="cuda") * 0.02])
    g = torch.randn(n, device="cuda").mul_(1e-3).to(torch.bfloat16)
    grp.step([g], HP)
    assert lmopt.optim_query_nonfinite(grp.handle) == 0
    g[:17] = float("inf")
    grp.step([g], HP)
    assert lmopt.optim_query_nonfinite(grp.handle) > 0
    with pytest.raises(lmopt.LmoptError) as e:
        lmopt.optim_step_nadam_kahan(grp.handle, [g.data_ptr()], 7, lmopt.NadamHparams(lr=1e-3, beta1=0.9, beta2=0.999), 0)
    assert e.value.code == lmopt.OPTIM_EINVAL
    bad = lmopt.NadamHparams(lr=1e-3, beta1=0.9, beta2=1.0, eps=1e-8)
    with pytest.raises(lmopt.LmoptError):
        lmopt.optim_step_nadam_kahan(grp.handle, [g.data_ptr()], 3, bad, 0)
    with pytest.raises(lmopt.LmoptError) as e:
        lmopt.optim_step_nadam_kahan(grp.handle, [g.data_ptr() + 1], 3, lmopt.NadamHparams(lr=1e-3, beta1=0.9, beta2=0.999), 0)
    assert e.value.code == lmopt.OPTIM_EALIGN


def test_deterministic_two_runs(eng):
    shapes = [(200_000,), (3000,)]
    outs = []
    for _ in range(2):
        masters = [W.master_weights(s, 9, i, device="cuda") for i, s in enumerate(shapes)]
        grp = eng.NadamGroup.from_masters(masters)
        for t in range(1, 4):
            grp.step([W.grad_bf16(s, 9, i, t, 1e-3, device="cuda") for i, s in enumerate(shapes)], HP)
        outs.append([x.clone() for x in grp.masters()] + [grp.m[0].clone(), grp.v[0].clone()])
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                           b.view(torch.int32) if b.dtype == torch.float32 else b)


@pytest.mark.parametrize("variant", ["nadamw", "adam"])
def test_f24_moments_bit_exact(orc, eng, variant):
    """f24 moment storage (NADAM_F24 groups): weights, residuals and both moment planes
    bit-identical to the oracle; sizes include fp32-moment tensors and ragged tails (the byte
    plane is padded to a 16-byte offset, so ragged sizes stay on the 128-bit path)."""
    sizes = [100, 4096, 4097, 16384, 16389, 40000, 131072]
    seed = 21
    hp = dict(HP, lr=1e-3, nesterov=variant.startswith("n"), weight_decay=0.02 if variant.endswith("w") else 0.0,
              wd_mode=1 if variant.endswith("w") else 0)
    masters = [W.master_weights((n,), seed, i) for i, n in enumerate(sizes)]
    ora = []
    for x in masters:
        hi, lo = orc.kahan_split(x.numpy())
        n = x.numel()
        st = ((np.zeros(n, np.float32), np.zeros(n, np.float32)) if n <= 4096 else
              (np.zeros(orc.f24_nbytes(n), np.uint8), np.zeros(orc.f24_nbytes(n), np.uint8)))
        ora.append(dict(hi=hi, lo=lo, m=st[0], v=st[1]))
    grp = eng.NadamGroup.from_masters([m.cuda() for m in masters], states="f24")
    mp = 1.0
    for t in range(1, 5):
        grads = [W.grad_bf16((n,), seed, i, t, 1e-3, zero_frac=0.01) for i, n in enumerate(sizes)]
        k, mp = orc.nadam_scalars(t, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"],
                                  hp["wd_mode"] == 1, hp["nesterov"], hp["momentum_decay"], mp)
        for o, g in zip(ora, grads):
            orc.nadam_step_tensor_f24(o["hi"], o["lo"], o["m"], o["v"], W.bits16(g), k)
        grp.step([g.cuda() for g in grads], hp)
    torch.cuda.synchronize()
    for i, o in enumerate(ora):
        assert np.array_equal(cuda_bits(grp.weights[i]), o["hi"]), i
        assert np.array_equal(cuda_bits(grp.res[i]), o["lo"]), i
        if sizes[i] <= 4096:
            assert np.array_equal(grp.m[i].cpu().numpy().view(np.uint32), o["m"].view(np.uint32))
            assert np.array_equal(grp.v[i].cpu().numpy().view(np.uint32), o["v"].view(np.uint32))
        else:
            assert np.array_equal(grp.m[i].cpu().numpy(), o["m"]), i
            assert np.array_equal(grp.v[i].cpu().numpy(), o["v"]), i


def test_f24_misaligned_buffers_take_scalar_path(orc, eng):
    """f24 groups whose buffers start 2 bytes past a 16-byte boundary go element by element and
    give the oracle's bits, padding bytes included."""
    from memory_lean_optimizer_gb300 import lmopt
    sizes = [5000, 20003]
    seed = 31
    masters = [W.master_weights((n,), seed, i) for i, n in enumerate(sizes)]
    keep, descs, dev, ora = [], [], [], []
    for i, n in enumerate(sizes):
        hi, lo = orc.kahan_split(masters[i].numpy())
        b1, w = alloc_offset(n, torch.int16, 1)
        b2, r = alloc_offset(n, torch.int16, 1)
        b3, m = alloc_offset(orc.f24_nbytes(n), torch.uint8, 2)
        b4, v = alloc_offset(orc.f24_nbytes(n), torch.uint8, 2)
        w.copy_(torch.from_numpy(hi.view(np.int16)))
        r.copy_(torch.from_numpy(lo.view(np.int16)))
        keep += [b1, b2, b3, b4]
        d = lmopt.TensorDesc(w_bf16=w.data_ptr(), res_u16=r.data_ptr(), m=m.data_ptr(), v=v.data_ptr(),
                             numel=n, ndim=1)
        d.shape[0] = n
        descs.append(d)
        dev.append((w, r, m, v))
        ora.append(dict(hi=hi, lo=lo, m=np.zeros(orc.f24_nbytes(n), np.uint8),
                        v=np.zeros(orc.f24_nbytes(n), np.uint8)))
    h = lmopt.optim_group_create(descs, lmopt.OPTIM_KIND_NADAM_F24)
    H = lmopt.NadamHparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, wd_mode=0,
                           nesterov=1, momentum_decay=0.004)
    mp = 1.0
    try:
        for t in range(1, 4):
            grads = [W.grad_bf16((n,), seed, i, t, 1e-3) for i, n in enumerate(sizes)]
            k, mp = orc.nadam_scalars(t, 1e-3, 0.9, 0.999, 1e-8, 0.0, False, True, 0.004, mp)
            for o, g in zip(ora, grads):
                orc.nadam_step_tensor_f24(o["hi"], o["lo"], o["m"], o["v"], W.bits16(g), k)
            gbufs = []
            for g in grads:
                b, gg = alloc_offset(g.numel(), torch.int16, 1)
                gg.copy_(g.view(torch.int16))
                gbufs += [b, gg]
            lmopt.optim_step_nadam_kahan(h, [gbufs[2 * i + 1].data_ptr() for i in range(len(sizes))], t, H, 0)
            torch.cuda.synchronize()
            for (w, r, m, v), o in zip(dev, ora):
                assert np.array_equal(cuda_bits(w), o["hi"])
                assert np.array_equal(cuda_bits(r), o["lo"])
                assert np.array_equal(m.cpu().numpy(), o["m"])
                assert np.array_equal(v.cpu().numpy(), o["v"])
    finally:
        lmopt.optim_group_destroy(h)


@pytest.mark.parametrize("states", ["u16", "f24"])
def test_stochastic_rounding_bit_exact(orc, eng, states):
    """Tensors without a residual and stochastic_rounding = 1: the stored bf16 weights follow the
    oracle's Philox4x32-10 draws bit for bit (vector and element-by-element paths)."""
    sizes = [300, 4097, 16384, 20003, 65536]
    seed, key = 23, 0xDEADBEEF12345
    hp = dict(HP, lr=1e-3, stochastic_rounding=1, seed=key)
    masters = [W.master_weights((n,), seed, i) for i, n in enumerate(sizes)]
    w0 = [m.to(torch.bfloat16) for m in masters]
    grp = eng.NadamGroup([w.cuda() for w in w0], kahan=False, states=states)
    ora = []
    for w in w0:
        n = w.numel()
        hi = W.bits16(w).copy()
        if n <= 4096:
            st = (np.zeros(n, np.float32), np.zeros(n, np.float32))
        elif states == "u16":
            st = (np.full(n, 32768, np.uint16), np.zeros(n, np.uint16))
        else:
            st = (np.zeros(orc.f24_nbytes(n), np.uint8), np.zeros(orc.f24_nbytes(n), np.uint8))
        ora.append(dict(hi=hi, m=st[0], v=st[1]))
    ost = orc.NadamState(len(sizes))
    mp = 1.0
    for t in range(1, 4):
        grads = [W.grad_bf16((n,), seed, i, t, 1e-3) for i, n in enumerate(sizes)]
        k, mp = orc.nadam_scalars(t, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], 0.0, False, True, 0.004, mp)
        for i, (o, g) in enumerate(zip(ora, grads)):
            if states == "u16":
                orc.nadam_step_tensor_sr(o["hi"], o["m"], o["v"], W.bits16(g), ost.scales[i], k, key, i, t)
            else:
                orc.nadam_step_tensor_f24(o["hi"], None, o["m"], o["v"], W.bits16(g), k, True, key, i, t)
        grp.step([g.cuda() for g in grads], hp)
        torch.cuda.synchronize()
        for i, o in enumerate(ora):
            assert np.array_equal(cuda_bits(grp.weights[i]), o["hi"]), (t, i)


def _degenerate_grad(kind, n, t, seed):
    """bf16 gradients for the degenerate cases (torch CPU, seeded)."""
    g = torch.Generator().manual_seed(1000 * seed + 10 * t + len(kind))
    x = torch.randn(n, generator=g)
    if kind == "zero_then_normal":          # exact zeros for two steps (zero scales), then normal
        x = x * 1e-3 if t > 2 else torch.zeros(n)
    elif kind == "subnormal":               # bf16 subnormals and zeros: squares underflow to 0
        x = x * 1e-39
        x[::3] = 0.0
    elif kind == "large":                   # |g| near 1e18: squares near 1e36, still finite
        x = x * 1e18
    elif kind == "two_scales":              # codes at both ends of the companding curve
        x = x * 1e-3
        x[: n // 2] *= 1e-27
    elif kind == "sign_flip":               # the same magnitudes, alternating sign per step
        x = x.abs() * 1e-3 * (1.0 if t % 2 else -1.0)
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("variant", ["nadamw", "adam_beta1_0", "lr_0"])
def test_degenerate_inputs_bit_exact(orc, eng, variant):
    """Degenerate inputs against the oracle, bit for bit after every step: all-zero gradients (the
    codec scales start at zero and stay there), bf16 subnormal gradients (squares underflow to
    zero; no flush to zero on either side), gradients near 1e18 (squares near the fp32 limit),
    two magnitude scales 27 decades apart in one tensor (codes at both ends of the curve), sign
    flips every step; u16 (> 4096 elements) and fp32 (<= 4096) tensors, ragged sizes.  Variants:
    NAdamW, Adam with beta1 = 0, and lr = 0 with decoupled decay (the weights stay bit for bit)."""
    kinds = ["zero_then_normal", "subnormal", "large", "two_scales", "sign_flip"]
    sizes = [20001, 3001, 16384, 70007, 4096]
    hp = dict(HP, lr=1e-3, weight_decay=0.01, wd_mode=1)
    if variant == "adam_beta1_0":
        hp = dict(hp, beta1=0.0, nesterov=0, weight_decay=0.0, wd_mode=0)
    elif variant == "lr_0":
        hp = dict(hp, lr=0.0)
    seed = 91
    shapes = [(n,) for n in sizes for _ in kinds]
    tkinds = [k for _ in sizes for k in kinds]
    masters = [W.master_weights(s, seed, i) for i, s in enumerate(shapes)]
    ora = OracleNadam(orc, [m.numpy() for m in masters])
    grp = eng.NadamGroup.from_masters([m.cuda() for m in masters])
    for t in range(1, 6):
        grads = [_degenerate_grad(k, s[0], t, seed + i) for i, (k, s) in enumerate(zip(tkinds, shapes))]
        ora.step([W.bits16(g).reshape(-1) for g in grads], hp)
        grp.step([g.cuda() for g in grads], hp)
        torch.cuda.synchronize()
        assert_nadam_equal(ora, grp, f"{variant} step {t}")
        for i, (a, b) in enumerate(zip(grp.scales(), ora.scales())):
            if W.numel(shapes[i]) > 4096:
                assert np.array_equal(np.float32(a), np.float32(b)), (t, i, tkinds[i], a, b)
    if variant == "lr_0":
        for i, m in enumerate(masters):
            hi, lo = orc.kahan_split(m.numpy().reshape(-1))
            assert np.array_equal(cuda_bits(grp.weights[i]).reshape(-1), hi)
    from memory_lean_optimizer_gb300 import lmopt
    assert lmopt.optim_query_nonfinite(grp.handle) == 0
    grp.close()


def test_verbose_banner(eng, capfd, monkeypatch):
    """LMOPT_VERBOSE=1: one stderr line per created group saying what is on; silent otherwise."""
    masters = [W.master_weights((n,), 5, i, device="cuda") for i, n in enumerate([5000, 300])]
    monkeypatch.setenv("LMOPT_VERBOSE", "1")
    grp = eng.NadamGroup.from_masters(masters)
    err = capfd.readouterr().err
    assert "lmopt: group of 2 tensors, 5300 elements, nadam u16 states, Kahan residual on 2 tensors" in err
    grp.close()
    monkeypatch.delenv("LMOPT_VERBOSE")
    grp = eng.NadamGroup.from_masters(masters)
    assert "lmopt:" not in capfd.readouterr().err
    grp.close()
