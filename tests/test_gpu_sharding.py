"""Tensors split across ranks, on one GPU: two groups hold the two ranks' slices of the same
tensors (plan_slices, world size 2).  Each step begins on both groups, takes the MAX of their
exchange buffers (what the all-reduce between two ranks computes), and ends on both.  Weights,
residuals and moment codes must equal the unsplit oracle step bit for bit.  (No kernel waits on
another here: the two groups' launches simply follow each other on one stream.)"""
import numpy as np
import pytest
import torch

from helpers import OracleNadam, cuda_bits
from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, wd_mode=1, nesterov=1,
          momentum_decay=0.004)
SIZES = [20000, 9000, 3000, 70001, 5000, 1 << 20]


@pytest.fixture(scope="module")
def eng():
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    return engine


def test_split_tensors_two_emulated_ranks(orc, eng):
    from memory_lean_optimizer_gb300.sharding import plan_slices, rank_slices
    seed = 9
    masters = [W.master_weights((n,), seed, i) for i, n in enumerate(SIZES)]
    ora = OracleNadam(orc, [m.numpy() for m in masters])
    full = [eng.kahan_split(m.cuda()) for m in masters]
    plan = plan_slices(SIZES, 2)
    assert sum(len(sl) > 1 for sl in plan) >= 3
    ranks = []
    for r in range(2):
        mine, ns = rank_slices(plan, r)
        grp = eng.NadamGroup([full[ti][0].view(-1)[a:b] for ti, a, b in mine],
                             [full[ti][1].view(-1)[a:b] for ti, a, b in mine])
        ranks.append((grp, mine, ns, grp.exchange_buffer()))
    ns = ranks[0][2]
    for t in range(1, 4):
        grads = [W.grad_bf16((n,), seed, i, t, 1e-3, zero_frac=0.01) for i, n in enumerate(SIZES)]
        ora.step([W.bits16(g) for g in grads], HP)
        gc = [g.cuda() for g in grads]
        for grp, mine, _, ex in ranks:
            grp.step_begin([gc[ti].view(-1)[a:b] for ti, a, b in mine], HP, ex)
        red = torch.maximum(ranks[0][3][: 3 * ns], ranks[1][3][: 3 * ns])
        for grp, _, _, ex in ranks:
            ex[: 3 * ns].copy_(red)
            grp.step_end(ex)
    torch.cuda.synchronize()
    for ti, (w, r) in enumerate(full):
        assert np.array_equal(cuda_bits(w).reshape(-1), ora.t[ti]["hi"]), f"tensor {ti}: weights differ"
        assert np.array_equal(cuda_bits(r).reshape(-1), ora.t[ti]["lo"]), f"tensor {ti}: residuals differ"
    for grp, mine, _, _ in ranks:
        for j, (ti, a, b) in enumerate(mine):
            m, v = ora.t[ti]["m"][a:b], ora.t[ti]["v"][a:b]
            if SIZES[ti] > 4096:
                assert np.array_equal(cuda_bits(grp.m[j]), m) and np.array_equal(cuda_bits(grp.v[j]), v), ti
            else:
                assert np.array_equal(grp.m[j].cpu().numpy().view(np.uint32), m.view(np.uint32)), ti
    for grp, *_ in ranks:
        grp.close()


def test_begin_end_states(eng):
    from memory_lean_optimizer_gb300 import lmopt
    grp = eng.NadamGroup.from_masters([torch.zeros(10000, device="cuda")])
    g = torch.zeros(10000, dtype=torch.bfloat16, device="cuda")
    ex = grp.exchange_buffer()
    with pytest.raises(lmopt.LmoptError, match="ESTATE"):
        grp.step_end(ex)
    grp.step_begin([g], HP, ex)
    with pytest.raises(lmopt.LmoptError, match="ESTATE"):
        grp.step_begin([g], HP, ex)
    with pytest.raises(lmopt.LmoptError, match="ESTATE"):
        lmopt.optim_group_set_step(grp.handle, 0, 1.0)
    grp.step_end(ex)
    grp.step([g], HP)          # the plain step still follows
    torch.cuda.synchronize()
    assert grp.step_count == 2 and torch.isfinite(ex).all()
    grp.close()
