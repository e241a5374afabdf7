"""GPU parity of the fused Adan step (m, v, n as fp32 planes or f24 buffers, the previous bf16
gradient, Kahan residual or stochastic rounding) against the oracle: bit-exact weights, residuals
and states."""
import numpy as np
import pytest
import torch

from helpers import cuda_bits
from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(lr=3.3e-5, beta1=0.02, beta2=0.08, beta3=0.01, eps=1e-8, weight_decay=0.02)


def _ora_state(orc, n, states):
    if states == "f24":
        return np.zeros(orc.adan_f24_nbytes(n), np.uint8)
    return np.zeros(3 * orc.adan_plane(n), np.float32)


def _ora_step(orc, states, o, g_bits, t, k, sr=False, seed=0, tensor=0):
    step = orc.adan_step_tensor_f24 if states == "f24" else orc.adan_step_tensor
    step(o["hi"], o["lo"], o["mnv"], o["gp"], g_bits, t, k, sr=sr, seed=seed, tensor=tensor)


def _state_bytes(t):
    return t.contiguous().cpu().view(torch.uint8).numpy()


@pytest.mark.parametrize("states", ["fp32", "f24"])
@pytest.mark.parametrize("rounding", ["kahan", "sr"])
def test_adan_bit_exact(orc, rounding, states):
    """fp32 states, or f24 states (three truncated 24-bit buffers above 4096 elements, fp32 planes
    at or below): weights, residuals, every stored state byte and the previous gradient equal the
    oracle's after each of 4 steps."""
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    # 128-bit path for every size (planes padded to 4 floats, f24 buffers to 16 bytes): whole
    # chunks, 8-element tails and sizes that are not multiples of 4 (1, 4097, 50001)
    sizes = [1, 100, 4096, 4097, 16384, 50001, 40004]
    seed, key = 50, 777
    hp = dict(HP, stochastic_rounding=int(rounding == "sr"), seed=key)
    masters = [W.master_weights((n,), seed, i) for i, n in enumerate(sizes)]
    if rounding == "kahan":
        grp = engine.AdanGroup.from_masters([m.cuda() for m in masters], states=states)
        ora = [dict(zip(("hi", "lo"), orc.kahan_split(m.numpy()))) for m in masters]
    else:
        grp = engine.AdanGroup([m.cuda().to(torch.bfloat16) for m in masters], kahan=False, states=states)
        ora = [dict(hi=W.bits16(m.to(torch.bfloat16)).copy(), lo=None) for m in masters]
    for o, n in zip(ora, sizes):
        o["mnv"] = _ora_state(orc, n, states)
        o["gp"] = np.zeros(n, np.uint16)
    k = orc.adan_scalars(hp["lr"], hp["beta1"], hp["beta2"], hp["beta3"], hp["eps"], hp["weight_decay"])
    for t in range(1, 5):
        grads = [W.grad_bf16((n,), seed, i, t, 1e-3, zero_frac=0.01) for i, n in enumerate(sizes)]
        for i, (o, g) in enumerate(zip(ora, grads)):
            _ora_step(orc, states, o, W.bits16(g), t, k, sr=rounding == "sr", seed=key, tensor=i)
        grp.step([g.cuda() for g in grads], hp)
        torch.cuda.synchronize()
        for i, o in enumerate(ora):
            assert np.array_equal(cuda_bits(grp.weights[i]), o["hi"]), (t, i)
            if o["lo"] is not None:
                assert np.array_equal(cuda_bits(grp.res[i]), o["lo"]), (t, i)
            assert np.array_equal(_state_bytes(grp.mvn[i]), o["mnv"].view(np.uint8)), (t, i)
            assert np.array_equal(cuda_bits(grp.gprev[i]), o["gp"]), (t, i)


def test_adan_f24_misaligned_buffers(orc):
    """f24 Adan states with a 2-byte (not 16-byte) aligned weight: the element-by-element path
    decodes and stores the three f24 buffers; results equal the oracle's bit for bit."""
    from helpers import alloc_offset
    from memory_lean_optimizer_gb300 import build, lmopt
    build.build()
    sizes = [5000, 9001]
    seed = 53
    keep, descs, ws, rs, bufs, gps, ora = [], [], [], [], [], [], []
    for i, n in enumerate(sizes):
        x = W.master_weights((n,), seed, i).numpy()
        hi, lo = orc.kahan_split(x)
        ora.append(dict(hi=hi, lo=lo, mnv=_ora_state(orc, n, "f24"), gp=np.zeros(n, np.uint16)))
        b1, w = alloc_offset(n, torch.int16, 1)
        b2, r = alloc_offset(n, torch.int16, 0)
        w.copy_(torch.from_numpy(hi.view(np.int16)))
        r.copy_(torch.from_numpy(lo.view(np.int16)))
        buf = torch.zeros(orc.adan_f24_nbytes(n), dtype=torch.uint8, device="cuda")
        gp = torch.zeros(n, dtype=torch.int16, device="cuda")
        keep += [b1, b2]
        ws.append(w), rs.append(r), bufs.append(buf), gps.append(gp)
        d = lmopt.TensorDesc(w_bf16=w.data_ptr(), res_u16=r.data_ptr(), m=buf.data_ptr(), v=gp.data_ptr(),
                             numel=n, ndim=1)
        d.shape[0] = n
        descs.append(d)
    h = lmopt.optim_group_create(descs, lmopt.OPTIM_KIND_ADAN_F24)
    H = lmopt.AdanHparams(lr=HP["lr"], beta1=HP["beta1"], beta2=HP["beta2"], beta3=HP["beta3"], eps=HP["eps"],
                          weight_decay=HP["weight_decay"])
    k = orc.adan_scalars(HP["lr"], HP["beta1"], HP["beta2"], HP["beta3"], HP["eps"], HP["weight_decay"])
    try:
        for t in range(1, 4):
            grads = [W.grad_bf16((n,), seed, i, t, 1e-3) for i, n in enumerate(sizes)]
            for i, (o, g) in enumerate(zip(ora, grads)):
                _ora_step(orc, "f24", o, W.bits16(g), t, k)
            gc = [g.cuda() for g in grads]
            lmopt.optim_step_adan(h, [g.data_ptr() for g in gc], t, H, 0)
            torch.cuda.synchronize()
        for i, o in enumerate(ora):
            assert np.array_equal(cuda_bits(ws[i]), o["hi"]) and np.array_equal(cuda_bits(rs[i]), o["lo"])
            assert np.array_equal(_state_bytes(bufs[i]), o["mnv"])
            assert np.array_equal(cuda_bits(gps[i]), o["gp"])
    finally:
        lmopt.optim_group_destroy(h)


def test_adan_empty_tensors(orc):
    """Tensors without elements among ordinary ones: the others follow the oracle bit for bit."""
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    sizes = [0, 4097, 0, 300]
    seed = 51
    masters = [W.master_weights((n,), seed, i) for i, n in enumerate(sizes)]
    grp = engine.AdanGroup.from_masters([m.cuda() for m in masters])
    ora = [dict(zip(("hi", "lo"), orc.kahan_split(m.numpy()))) for m in masters]
    for o, n in zip(ora, sizes):
        o["mnv"] = np.zeros(3 * orc.adan_plane(n), np.float32)
        o["gp"] = np.zeros(n, np.uint16)
    k = orc.adan_scalars(HP["lr"], HP["beta1"], HP["beta2"], HP["beta3"], HP["eps"], HP["weight_decay"])
    for t in range(1, 4):
        grads = [W.grad_bf16((n,), seed, i, t, 1e-3) for i, n in enumerate(sizes)]
        for i, (o, g) in enumerate(zip(ora, grads)):
            if sizes[i]:
                orc.adan_step_tensor(o["hi"], o["lo"], o["mnv"], o["gp"], W.bits16(g), t, k)
        grp.step([g.cuda() for g in grads], HP)
    torch.cuda.synchronize()
    for i, o in enumerate(ora):
        if sizes[i]:
            assert np.array_equal(cuda_bits(grp.weights[i]), o["hi"]) and np.array_equal(cuda_bits(grp.res[i]), o["lo"])


@pytest.mark.parametrize("states", ["fp32", "f24"])
def test_adan_degenerate_inputs_bit_exact(orc, states):
    """Degenerate gradients against the oracle, every byte after each of 5 steps: all zeros for two
    steps then normal, bf16 subnormals (squares underflow), magnitudes near 1e18 (c c near the
    fp32 limit), two scales 27 decades apart in one tensor, a sign flip every step (large
    differences d = g - g_prev); fp32-plane (<= 4096) and f24 tensors."""
    from test_gpu_nadam import _degenerate_grad
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    kinds = ["zero_then_normal", "subnormal", "large", "two_scales", "sign_flip"]
    sizes = [3001, 20001]
    seed = 97
    shapes = [n for n in sizes for _ in kinds]
    tkinds = [k for _ in sizes for k in kinds]
    masters = [W.master_weights((n,), seed, i) for i, n in enumerate(shapes)]
    grp = engine.AdanGroup.from_masters([m.cuda() for m in masters], states=states)
    ora = [dict(zip(("hi", "lo"), orc.kahan_split(m.numpy()))) for m in masters]
    for o, n in zip(ora, shapes):
        o["mnv"] = _ora_state(orc, n, states)
        o["gp"] = np.zeros(n, np.uint16)
    k = orc.adan_scalars(HP["lr"], HP["beta1"], HP["beta2"], HP["beta3"], HP["eps"], HP["weight_decay"])
    for t in range(1, 6):
        grads = [_degenerate_grad(kd, n, t, seed + i) for i, (kd, n) in enumerate(zip(tkinds, shapes))]
        for o, g in zip(ora, grads):
            _ora_step(orc, states, o, W.bits16(g), t, k)
        grp.step([g.cuda() for g in grads], HP)
        torch.cuda.synchronize()
        for i, o in enumerate(ora):
            tag = (t, i, tkinds[i], shapes[i])
            assert np.array_equal(cuda_bits(grp.weights[i]), o["hi"]), tag
            assert np.array_equal(cuda_bits(grp.res[i]), o["lo"]), tag
            assert np.array_equal(_state_bytes(grp.mvn[i]), o["mnv"].view(np.uint8)), tag
            assert np.array_equal(cuda_bits(grp.gprev[i]), o["gp"]), tag
    from memory_lean_optimizer_gb300 import lmopt
    assert lmopt.optim_query_nonfinite(grp.handle) == 0
    grp.close()
