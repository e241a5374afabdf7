"""GPU parity of the fused Adan step (fp32 m, v, n and the previous bf16 gradient, Kahan residual
or stochastic rounding) against the oracle: bit-exact weights, residuals and states."""
import numpy as np
import pytest
import torch

from helpers import cuda_bits
from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(lr=3.3e-5, beta1=0.02, beta2=0.08, beta3=0.01, eps=1e-8, weight_decay=0.02)


@pytest.mark.parametrize("rounding", ["kahan", "sr"])
def test_adan_bit_exact(orc, rounding):
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    # 128-bit path for every size (planes padded to 4 floats): whole chunks, 8-element tails and
    # sizes that are not multiples of 4 (1, 4097, 50001)
    sizes = [1, 100, 4097, 16384, 50001, 40004]
    seed, key = 50, 777
    hp = dict(HP, stochastic_rounding=int(rounding == "sr"), seed=key)
    masters = [W.master_weights((n,), seed, i) for i, n in enumerate(sizes)]
    if rounding == "kahan":
        grp = engine.AdanGroup.from_masters([m.cuda() for m in masters])
        ora = [dict(zip(("hi", "lo"), orc.kahan_split(m.numpy()))) for m in masters]
    else:
        grp = engine.AdanGroup([m.cuda().to(torch.bfloat16) for m in masters], kahan=False)
        ora = [dict(hi=W.bits16(m.to(torch.bfloat16)).copy(), lo=None) for m in masters]
    for o, n in zip(ora, sizes):
        o["mnv"] = np.zeros(3 * orc.adan_plane(n), np.float32)
        o["gp"] = np.zeros(n, np.uint16)
    k = orc.adan_scalars(hp["lr"], hp["beta1"], hp["beta2"], hp["beta3"], hp["eps"], hp["weight_decay"])
    for t in range(1, 5):
        grads = [W.grad_bf16((n,), seed, i, t, 1e-3, zero_frac=0.01) for i, n in enumerate(sizes)]
        for i, (o, g) in enumerate(zip(ora, grads)):
            orc.adan_step_tensor(o["hi"], o["lo"], o["mnv"], o["gp"], W.bits16(g), t, k,
                                 sr=rounding == "sr", seed=key, tensor=i)
        grp.step([g.cuda() for g in grads], hp)
        torch.cuda.synchronize()
        for i, o in enumerate(ora):
            assert np.array_equal(cuda_bits(grp.weights[i]), o["hi"]), (t, i)
            if o["lo"] is not None:
                assert np.array_equal(cuda_bits(grp.res[i]), o["lo"]), (t, i)
            assert np.array_equal(grp.mvn[i].cpu().numpy().view(np.uint32), o["mnv"].view(np.uint32)), (t, i)
            assert np.array_equal(cuda_bits(grp.gprev[i]), o["gp"]), (t, i)


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
