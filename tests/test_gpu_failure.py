"""Failure handling of the host side, on a GPU, without a GPU fault: a bounded host wait that runs
out (made to run out at once by the host-side injection LMOPT_FAULT_INJECT=timeout) returns
OPTIM_ETIMEOUT, leaves weights, states and counters untouched, and the same call succeeds once
the wait can complete.  Nothing is made to hang, trap or fault on the device."""
import numpy as np
import pytest
import torch

from helpers import OracleNadam, assert_nadam_equal
from memory_lean_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(W.NADAM_HP, lr=1e-3)


def test_injected_wait_timeout_leaves_state_untouched(orc, monkeypatch):
    from memory_lean_optimizer_gb300 import build, engine, lmopt
    build.build()
    shapes = [(3000,), (70001,), (256, 96)]
    seed = 61
    masters = [W.master_weights(s, seed, i) for i, s in enumerate(shapes)]
    ora = OracleNadam(orc, [m.numpy() for m in masters])
    grp = engine.NadamGroup.from_masters([m.cuda() for m in masters])
    g1 = [W.grad_bf16(s, seed, i, 1, 1e-3) for i, s in enumerate(shapes)]
    g1c = [g.cuda() for g in g1]
    ora.step([W.bits16(g).reshape(-1) for g in g1], HP)
    grp.step(g1c, HP)
    torch.cuda.synchronize()
    before = [t.clone() for t in grp.weights + grp.res + grp.m + grp.v]
    g2 = [W.grad_bf16(s, seed, i, 2, 1e-3) for i, s in enumerate(shapes)]
    g2c = [g.cuda() for g in g2]          # new device pointers: the step must upload them (a wait)

    monkeypatch.setenv("LMOPT_FAULT_INJECT", "timeout")
    for call in (lambda: lmopt.optim_query_scales(grp.handle, len(shapes)),
                 lambda: lmopt.optim_query_nonfinite(grp.handle),
                 lambda: grp.step(g2c, HP)):
        with pytest.raises(lmopt.LmoptError) as e:
            call()
        assert e.value.code == lmopt.OPTIM_ETIMEOUT, e.value
        assert "injected timeout" in str(e.value)
    monkeypatch.delenv("LMOPT_FAULT_INJECT")
    torch.cuda.synchronize()
    assert lmopt.optim_group_get_step(grp.handle)[0] == 1
    after = grp.weights + grp.res + grp.m + grp.v
    assert all(torch.equal(a, b) for a, b in zip(before, after))

    grp.step(g2c, HP)                     # the same call now succeeds
    ora.step([W.bits16(g).reshape(-1) for g in g2], HP)
    torch.cuda.synchronize()
    assert_nadam_equal(ora, grp, "after the timed-out step")
    got = lmopt.optim_query_scales(grp.handle, len(shapes))
    for i, (a, b) in enumerate(zip(got, ora.scales())):
        if W.numel(shapes[i]) > 4096:
            assert np.array_equal(np.float32(a), np.float32(b)), (i, a, b)
    assert lmopt.optim_query_nonfinite(grp.handle) == 0
    grp.close()
