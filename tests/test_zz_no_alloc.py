"""The allocation-free factored step, called through the C ABI, against the regular entry point.

Some callers cannot call cudaMalloc (their device memory belongs to another allocator or a fixed
pool, or they must not allocate once set up), so optim_step_factored_noalloc keeps all of its
scratch in one fixed device array instead of allocating per group.  Its results must match
optim_step_factored on a group holding the same single tensor, over two calls in a row (the
second call runs on the array the first one left behind).  This file is collected last so that a
run stopping at the first failure has already run every other test; it also passes alone.
"""
import numpy as np
import pytest
import torch

from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta2=0.999, decay_rate=-0.8, eps1=1e-30, eps2=1e-30, d=1.0, clip_threshold=1.0,
          weight_decay=0.01, mode=0)


def _hparams(lmopt, hp):
    return lmopt.FactoredHparams(lr=hp["lr"], beta2=hp["beta2"], decay_rate=hp["decay_rate"], eps1=hp["eps1"],
                                 eps2=hp["eps2"], d=hp["d"], clip_threshold=hp["clip_threshold"],
                                 weight_decay=hp["weight_decay"], mode=hp["mode"])


PRODIGY_FIXED_D = dict(HP, mode=1, beta2=0.99, d=0.37)   # Prodigy mode with a fixed d != 1


@pytest.mark.parametrize("hp", [HP, PRODIGY_FIXED_D], ids=["adafactor", "prodigy-fixed-d"])
@pytest.mark.parametrize("shape", [(300, 257), (1024, 640), (8, 8, 3, 3), (5000,)])
def test_noalloc_matches_group_step_two_calls(shape, hp):
    from memory_lean_optimizer_gb300 import build, engine, lmopt
    build.build()
    master = W.master_weights(shape, 7, 0, device="cuda")
    ref = engine.FactoredGroup.from_masters([master.clone()])      # regular entry point
    alt = engine.FactoredGroup.from_masters([master.clone()])      # buffers for the no-alloc calls
    d = engine._desc(alt.weights[0], alt.res[0], alt.row[0], alt.col[0], shape)
    h = _hparams(lmopt, hp)
    stream = torch.cuda.current_stream().cuda_stream
    for step in (1, 2):
        g = W.grad_bf16(shape, 7, 0, step, 1e-3, device="cuda")
        ref.step([g], hp)
        lmopt.optim_step_factored_noalloc(d, g.data_ptr(), step, h, stream)
        torch.cuda.synchronize()
        # same tolerance as the factored parity tests: masters 1e-6 relative + 1e-6 lr per step,
        # statistics 1e-6 relative (the two paths run the same kernels, so they agree exactly)
        a = ref.masters()[0].double()
        b = alt.masters()[0].double()
        assert torch.all((a - b).abs() <= 1e-6 * a.abs() + 1e-6 * hp["lr"] * hp["d"] * step)
        for x, y in ((ref.row[0], alt.row[0]), (ref.col[0], alt.col[0])):
            if x is not None:
                assert torch.all((x.double() - y.double()).abs() <= 1e-6 * x.double().abs() + 1e-37)
    assert torch.equal(ref.weights[0].view(torch.int16), alt.weights[0].view(torch.int16))
    ref.close()
    alt.close()


def test_noalloc_rejects_oversized_tensor():
    from memory_lean_optimizer_gb300 import lmopt
    d = lmopt.TensorDesc(w_bf16=0x100000, res_u16=0x200000, m=0x300000, v=0x400000, numel=100_000 * 100_000, ndim=2)
    d.shape[0], d.shape[1] = 100_000, 100_000
    with pytest.raises(lmopt.LmoptError) as e:
        lmopt.optim_step_factored_noalloc(d, 0x500000, 1, _hparams(lmopt, HP), 0)
    assert e.value.code == lmopt.OPTIM_EINVAL
    assert "scratch" in str(e.value)


def test_noalloc_checks_hyper_parameters_like_the_group_step():
    """Non-finite eps1 or eps2 (or a negative one) is rejected before anything is enqueued, as by
    optim_step_factored."""
    from memory_lean_optimizer_gb300 import lmopt
    d = lmopt.TensorDesc(w_bf16=0x100000, res_u16=0x200000, m=0x300000, v=0x400000, numel=64 * 64, ndim=2)
    d.shape[0], d.shape[1] = 64, 64
    for bad in (dict(HP, eps1=float("inf")), dict(HP, eps2=float("inf")), dict(HP, eps1=-1e-30),
                dict(PRODIGY_FIXED_D, d=float("inf"))):
        with pytest.raises(lmopt.LmoptError) as e:
            lmopt.optim_step_factored_noalloc(d, 0x500000, 1, _hparams(lmopt, bad), 0)
        assert e.value.code == lmopt.OPTIM_EINVAL and "hyper-parameters" in str(e.value)
