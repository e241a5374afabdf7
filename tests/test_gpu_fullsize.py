"""Parity at full workload sizes, in the launch configuration the benchmark times (one library
group per Flux-like block, the ten SDXL-like factored groups, one group of 20,000 ragged tensors, the
35-group host-offload pipeline), each for its configuration's own number of steps (5, and 3 for the
offload pipeline), and the NEXT rows (f24 moments, stochastic rounding, Adan with fp32 and f24
states) on the flux19 workload for its 5 steps.  Every tensor of every workload is replayed by
the oracle: flux19 and ragged20k after step 1 and after their last step, the others after their
last step.  The oracle replays tensor by tensor on a thread pool (one single-threaded oracle call
per tensor), each tensor's inputs regenerated from their seeds on the device and copied back, so
host memory stays bounded by the tensors in flight."""
import os
from collections import deque
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from helpers import OracleNadam
from memory_lean_optimizer_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.full]


@pytest.fixture(scope="module")
def eng():
    from memory_lean_optimizer_gb300 import build, engine
    build.build()
    return engine


def _bits(t):
    return W.bits16(t).reshape(-1)


def _f32(t):
    return t.detach().contiguous().cpu().numpy().reshape(-1)


class Replays:
    """Oracle replays of single tensors on every host core, at most `depth` in flight; a failed
    comparison is raised by submit() or finish()."""

    def __init__(self):
        workers = os.cpu_count() or 4
        self.pool = ThreadPoolExecutor(max_workers=workers)
        self.depth = workers + 4
        self.futs = deque()
        self.done = 0

    def submit(self, fn, *args):
        while len(self.futs) >= self.depth:
            self.futs.popleft().result()
            self.done += 1
        self.futs.append(self.pool.submit(fn, *args))

    def finish(self):
        while self.futs:
            self.futs.popleft().result()
            self.done += 1
        self.pool.shutdown()
        return self.done


def _replay_nadam(orc, x, grads, hp, got, scale, tag):
    """One tensor's NAdam trajectory in the oracle, compared bit for bit with the GPU's state
    (weights, residuals, u16 codes or fp32 moments, scale record)."""
    o = OracleNadam(orc, [x])
    for g in grads:
        o.step([g], hp)
    ot = o.t[0]
    for key in ("hi", "lo", "m", "v"):
        want = ot[key].view(np.uint8) if ot[key].dtype == np.float32 else ot[key]
        have = got[key].view(np.uint8) if got[key].dtype == np.float32 else got[key]
        if not np.array_equal(have, want):
            bad = np.flatnonzero(have != want)
            raise AssertionError(f"{tag}: {key} differs in {bad.size} places, first {bad[:5]}")
    if x.size > 4096:
        assert np.array_equal(np.float32(scale), np.float32(o.scales()[0])), f"{tag}: scale record {scale} != {o.scales()[0]}"


def _nadam_state(grp, i):
    n = grp.weights[i].numel()
    if n > 4096:
        m, v = _bits(grp.m[i]), _bits(grp.v[i])
    else:
        m, v = _f32(grp.m[i]), _f32(grp.v[i])
    return dict(hi=_bits(grp.weights[i]), lo=_bits(grp.res[i]), m=m, v=v)


def _check_nadam_groups(orc, groups, shapes_per_group, tids, cfg, upto, tag):
    """Every tensor of every group after `upto` steps against the oracle."""
    from memory_lean_optimizer_gb300 import lmopt
    rp = Replays()
    for b, (grp, shapes) in enumerate(zip(groups, shapes_per_group)):
        scales = lmopt.optim_query_scales(grp.handle, len(shapes))
        for i, s in enumerate(shapes):
            tid = tids[b][i]
            x = _f32(W.master_weights(s, cfg["seed"], tid, device="cuda"))
            gs = [_bits(W.grad_bf16(s, cfg["seed"], tid, t, cfg["g_std"], device="cuda", zero_frac=cfg["zero_frac"]))
                  for t in range(1, upto + 1)]
            rp.submit(_replay_nadam, orc, x, gs, cfg["hp"], _nadam_state(grp, i), scales[i],
                      f"{tag} step {upto} group {b} tensor {i} {tuple(s)}")
        assert lmopt.optim_query_nonfinite(grp.handle) == 0
    return rp.finish()


def _run_nadam_workload(orc, eng, name):
    cfg = W.config(name)
    steps = cfg["steps"]
    groups, tids, tid = [], [], 0
    for shapes in cfg["groups"]:
        ids = list(range(tid, tid + len(shapes)))
        masters = [W.master_weights(s, cfg["seed"], j, device="cuda") for s, j in zip(shapes, ids)]
        groups.append(eng.NadamGroup.from_masters(masters))
        del masters
        tids.append(ids)
        tid += len(shapes)

    def gpu_step(t):
        for grp, shapes, ids in zip(groups, cfg["groups"], tids):
            grads = [W.grad_bf16(s, cfg["seed"], j, t, cfg["g_std"], device="cuda", zero_frac=cfg["zero_frac"])
                     for s, j in zip(shapes, ids)]
            grp.step(grads, cfg["hp"])
            del grads

    gpu_step(1)
    torch.cuda.synchronize()
    n1 = _check_nadam_groups(orc, groups, cfg["groups"], tids, cfg, 1, name)
    for t in range(2, steps + 1):
        gpu_step(t)
    torch.cuda.synchronize()
    n2 = _check_nadam_groups(orc, groups, cfg["groups"], tids, cfg, steps, name)
    assert n1 == n2 == tid
    for grp in groups:
        grp.close()
    del groups
    torch.cuda.empty_cache()


def test_flux19_full(orc, eng):
    """19 blocks x 5 Flux-like linears (3,227,516,928 params), NAdamW wd 0.01, 5 steps, one group
    per block: all 95 tensors bit-identical to the oracle after step 1 and after step 5."""
    _run_nadam_workload(orc, eng, "flux19")


def test_ragged20k_full(orc, eng):
    """20,000 tensors (sizes round(2^U(6,22)), ~7.56e9 params, 37.5% with fp32 moments), 1%
    exact-zero gradients, one group, 5 steps: every tensor bit-identical to the oracle after step 1
    and after step 5."""
    _run_nadam_workload(orc, eng, "ragged20k")


def _replay_factored(orc, x, shape, grads, hp, got_master, got_states, tag):
    from test_gpu_factored import OracleFactored
    o = OracleFactored(orc, [x], [shape])
    for g in grads:
        o.step([g], hp)
    ot = o.t[0]
    steps = len(grads)
    ref = orc.kahan_merge(ot["hi"], ot["lo"]).astype(np.float64)
    got = got_master.astype(np.float64)
    tol = 1e-6 * np.abs(ref) + 1e-6 * hp["lr"] * steps
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{tag}: {bad.sum()} masters out of tolerance"
    names = ("row", "col") if "row" in ot else ("V",)
    for name, st in zip(names, got_states):
        r = ot[name].astype(np.float64)
        assert np.all(np.abs(st.astype(np.float64) - r) <= 1e-6 * np.abs(r) + 1e-37), f"{tag}: {name} state differs"


def test_sdxl_like_full(orc, eng):
    """SDXL-like factored workload (1332 tensors, 2,602,705,920 params) in its 10 groups,
    Adafactor mode, 5 steps: every tensor's fp32 master within 1e-6 relative (+1e-6 lr per step)
    and its row/column (or 1-D) statistics within 1e-6 relative of the oracle."""
    cfg = W.config("sdxl_like")
    hp, steps = cfg["hp"], cfg["steps"]
    shapes = [s for g in cfg["groups"] for s in g]
    bounds = np.cumsum([0] + [len(g) for g in cfg["groups"]])
    groups = []
    for k in range(len(cfg["groups"])):
        masters = [W.master_weights(shapes[i], 0, i, device="cuda") for i in range(bounds[k], bounds[k + 1])]
        groups.append(eng.FactoredGroup.from_masters(masters))
        del masters
    for t in range(1, steps + 1):
        for k, grp in enumerate(groups):
            grads = [W.grad_bf16(shapes[i], 0, i, t, cfg["g_std"], device="cuda") for i in range(bounds[k], bounds[k + 1])]
            grp.step(grads, hp)
            del grads
    torch.cuda.synchronize()
    rp = Replays()
    from memory_lean_optimizer_gb300 import lmopt
    for k, grp in enumerate(groups):
        masters = grp.masters()
        for li, i in enumerate(range(bounds[k], bounds[k + 1])):
            s = shapes[i]
            x = _f32(W.master_weights(s, 0, i, device="cuda"))
            gs = [_bits(W.grad_bf16(s, 0, i, t, cfg["g_std"], device="cuda")) for t in range(1, steps + 1)]
            states = [_f32(grp.row[li]), _f32(grp.col[li])] if grp.row[li] is not None else [_f32(grp.col[li])]
            rp.submit(_replay_factored, orc, x, tuple(s), gs, hp, _f32(masters[li]), states,
                      f"sdxl_like step {steps} tensor {i} {tuple(s)}")
        del masters
        assert lmopt.optim_query_nonfinite(grp.handle) == 0
    assert rp.finish() == len(shapes)
    for grp in groups:
        grp.close()
    del groups
    torch.cuda.empty_cache()


def test_flux35_offload_full(orc, eng):
    """35 Flux-like blocks (5,945,425,920 params) with residuals and u16 moments in pinned host
    memory (35.7 GB), 3 staging slots, 3 steps: every tensor bit-identical to the oracle."""
    cfg = W.config("flux35")
    hp, steps = cfg["hp"], cfg["steps"]
    shapes = cfg["groups"][0]
    slot = eng.offload_slot_bytes([W.numel(s) for s in shapes])
    off = eng.OffloadEngine(slot, 3)
    groups = []
    for b in range(35):
        masters = [W.master_weights(s, 0, 1000 * b + i, device="cuda") for i, s in enumerate(shapes)]
        groups.append(eng.NadamGroup.from_masters(masters, offload=off))
        del masters
    host_grads = []
    for t in range(1, steps + 1):
        grads = [W.grad_bf16(s, 0, i, t, cfg["g_std"], device="cuda") for i, s in enumerate(shapes)]
        host_grads.append([_bits(g) for g in grads])
        groups[0].prefetch()
        for k, grp in enumerate(groups):
            if k + 1 < len(groups):
                groups[k + 1].prefetch()
            grp.step(grads, hp)
        del grads
    off.sync()
    torch.cuda.synchronize()
    from memory_lean_optimizer_gb300 import lmopt
    rp = Replays()
    for b, grp in enumerate(groups):
        scales = lmopt.optim_query_scales(grp.handle, len(shapes))
        for i, s in enumerate(shapes):
            x = _f32(W.master_weights(s, 0, 1000 * b + i, device="cuda"))
            got = dict(hi=_bits(grp.weights[i]), lo=grp.res[i].numpy().view(np.uint16).reshape(-1).copy(),
                       m=grp.m[i].numpy().view(np.uint16).reshape(-1).copy(),
                       v=grp.v[i].numpy().view(np.uint16).reshape(-1).copy())
            rp.submit(_replay_nadam, orc, x, [hg[i] for hg in host_grads], hp, got, scales[i],
                      f"flux35 step {steps} block {b} tensor {i}")
    assert rp.finish() == 35 * len(shapes)
    for g in groups:
        g.close()
    off.close()
    del groups
    torch.cuda.empty_cache()


def test_tensor_beyond_2_31_elements(orc, eng):
    """One tensor of 2^31 + 13 elements (64-bit element offsets, 65,537 chunks), one NAdamW
    step: sampled elements -- chunk edges, both sides of 2^31, the last one, random ones -- equal
    the oracle's step of the same element, given the tensor's max|g| computed on the host."""
    n = (1 << 31) + 13
    hp = dict(W.NADAM_HP, weight_decay=0.01, wd_mode=1)
    master = W.master_weights((n,), 3, 0, device="cuda")
    grp = eng.NadamGroup.from_masters([master])
    rng = np.random.default_rng(0)
    idx = np.unique(np.concatenate([[0, 1, 7, 8, 16383, 16384, 32767, 32768, (1 << 31) - 1, 1 << 31, (1 << 31) + 5, n - 1],
                                    rng.integers(0, n, 200)]))
    it = torch.from_numpy(idx).cuda()
    x = master[it].cpu().numpy()
    del master
    torch.cuda.empty_cache()
    g = W.grad_bf16((n,), 3, 0, 1, 1e-4, device="cuda")
    gmax = 0
    for c in range(0, n, 1 << 28):          # max |g| on the host, in pieces
        part = W.bits16(g[c:c + (1 << 28)]) & 0x7FFF
        gmax = max(gmax, int(part.max()))
    G = float(np.array([gmax << 16], np.uint32).view(np.float32)[0])
    gs = W.bits16(g[it])
    grp.step([g], hp)
    torch.cuda.synchronize()
    got = {name: W.bits16(t[it]) for name, t in (("hi", grp.weights[0]), ("lo", grp.res[0]), ("m", grp.m[0]), ("v", grp.v[0]))}
    k, _ = orc.nadam_scalars(1, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], True, True,
                             hp["momentum_decay"], 1.0)
    for j in range(idx.size):
        hi, lo = orc.kahan_split(x[j:j + 1])
        m, v = np.full(1, 32768, np.uint16), np.zeros(1, np.uint16)
        sc = orc.Scale()
        orc.nadam_step_slice(hi, lo, m, v, gs[j:j + 1], False, G, sc, k)
        for name, want in (("hi", hi), ("lo", lo), ("m", m), ("v", v)):
            assert got[name][j] == want[0], f"element {idx[j]}: {name} {got[name][j]} != {want[0]}"
    grp.close()
    del g, grp
    torch.cuda.empty_cache()


ADAN_HP = dict(lr=3.3e-5, beta1=0.02, beta2=0.08, beta3=0.01, eps=1e-8, weight_decay=0.02)
SR_SEED = 12345
NEXT_STEPS = 5          # the flux19 configuration's step count


def _replay_next(orc, variant, x, grads, hp, got, tensor, scale, tag):
    """One tensor's trajectory under a NEXT-row variant, bit for bit against the GPU's bytes."""
    n = x.size
    if variant == "sr":
        o = dict(hi=orc.round_bf16(x), lo=None)
    else:
        hi, lo = orc.kahan_split(x)
        o = dict(hi=hi, lo=lo)
    if variant in ("f24", "sr"):
        small = n <= 4096
        if small:
            o["m"], o["v"] = np.zeros(n, np.float32), np.zeros(n, np.float32)
        elif variant == "f24":
            o["m"], o["v"] = np.zeros(orc.f24_nbytes(n), np.uint8), np.zeros(orc.f24_nbytes(n), np.uint8)
        else:
            o["m"], o["v"] = np.full(n, 32768, np.uint16), np.zeros(n, np.uint16)
        sc, mp = orc.Scale(), 1.0
        for t, g in enumerate(grads, start=1):
            k, mp = orc.nadam_scalars(t, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"],
                                      hp["wd_mode"] == 1, hp["nesterov"], hp["momentum_decay"], mp)
            if variant == "f24":
                orc.nadam_step_tensor_f24(o["hi"], o["lo"], o["m"], o["v"], g, k)
            else:
                orc.nadam_step_tensor_sr(o["hi"], o["m"], o["v"], g, sc, k, SR_SEED, tensor, t)
        keys = ("hi", "m", "v") if variant == "sr" else ("hi", "lo", "m", "v")
        if variant == "sr" and n > 4096:
            assert np.array_equal(np.float32(scale), np.float32((sc.s_m, sc.s_v, sc.a_m, sc.a_v))), f"{tag}: scale record"
    else:
        k = orc.adan_scalars(hp["lr"], hp["beta1"], hp["beta2"], hp["beta3"], hp["eps"], hp["weight_decay"])
        o["mnv"] = (np.zeros(orc.adan_f24_nbytes(n), np.uint8) if variant == "adan_f24"
                    else np.zeros(3 * orc.adan_plane(n), np.float32))
        o["gp"] = np.zeros(n, np.uint16)
        step = orc.adan_step_tensor_f24 if variant == "adan_f24" else orc.adan_step_tensor
        for t, g in enumerate(grads, start=1):
            step(o["hi"], o["lo"], o["mnv"], o["gp"], g, t, k)
        keys = ("hi", "lo", "mnv", "gp")
    for key in keys:
        want = np.ascontiguousarray(o[key]).view(np.uint8)
        have = np.ascontiguousarray(got[key]).view(np.uint8)
        if not np.array_equal(have, want):
            bad = np.flatnonzero(have != want)
            raise AssertionError(f"{tag}: {key} differs in {bad.size} bytes, first {bad[:5]}")


def _bytes(t):
    return t.detach().contiguous().cpu().view(torch.uint8).numpy().reshape(-1)


@pytest.mark.parametrize("variant", ["f24", "sr", "adan", "adan_f24"])
def test_flux19_next_rows_full(orc, eng, variant):
    """The NEXT rows at the headline workload's size, in the benchmark's launch configuration (one
    group per Flux-like block, 19 groups, 3,227,516,928 params), 5 steps: NAdamW with f24
    moments; u16 moments with stochastic rounding instead of the residual; Adan with fp32 states;
    Adan with f24 states.  Every tensor's weights, residuals and every stored state byte equal the
    oracle's replay of that tensor."""
    from memory_lean_optimizer_gb300 import lmopt
    cfg = W.config("flux19")
    nadam = variant in ("f24", "sr")
    hp = dict(cfg["hp"], stochastic_rounding=int(variant == "sr"), seed=SR_SEED) if nadam else dict(ADAN_HP)
    groups, tids, tid = [], [], 0
    for shapes in cfg["groups"]:
        ids = list(range(tid, tid + len(shapes)))
        masters = [W.master_weights(s, cfg["seed"], j, device="cuda") for s, j in zip(shapes, ids)]
        if variant == "f24":
            groups.append(eng.NadamGroup.from_masters(masters, states="f24"))
        elif variant == "sr":
            groups.append(eng.NadamGroup([x.to(torch.bfloat16) for x in masters], kahan=False))
        else:
            groups.append(eng.AdanGroup.from_masters(masters, states="f24" if variant == "adan_f24" else "fp32"))
        del masters
        tids.append(ids)
        tid += len(shapes)
    for t in range(1, NEXT_STEPS + 1):
        for grp, shapes, ids in zip(groups, cfg["groups"], tids):
            grads = [W.grad_bf16(s, cfg["seed"], j, t, cfg["g_std"], device="cuda") for s, j in zip(shapes, ids)]
            grp.step(grads, hp)
            del grads
    torch.cuda.synchronize()
    rp = Replays()
    for b, (grp, shapes) in enumerate(zip(groups, cfg["groups"])):
        scales = lmopt.optim_query_scales(grp.handle, len(shapes)) if variant == "sr" else [None] * len(shapes)
        for i, s in enumerate(shapes):
            j = tids[b][i]
            x = _f32(W.master_weights(s, cfg["seed"], j, device="cuda"))
            gs = [_bits(W.grad_bf16(s, cfg["seed"], j, t, cfg["g_std"], device="cuda")) for t in range(1, NEXT_STEPS + 1)]
            got = dict(hi=_bytes(grp.weights[i]))
            if variant != "sr":
                got["lo"] = _bytes(grp.res[i])
            if nadam:
                got["m"], got["v"] = _bytes(grp.m[i]), _bytes(grp.v[i])
            else:
                got["mnv"], got["gp"] = _bytes(grp.mvn[i]), _bytes(grp.gprev[i])
            rp.submit(_replay_next, orc, variant, x, gs, hp, got, i, scales[i],
                      f"flux19 {variant} step {NEXT_STEPS} group {b} tensor {i} {tuple(s)}")
        assert lmopt.optim_query_nonfinite(grp.handle) == 0
    assert rp.finish() == tid
    for grp in groups:
        grp.close()
    del groups
    torch.cuda.empty_cache()


def test_sdxl_like_prodigy_full(orc, eng):
    """NEXT-4 at full size, in the benchmark's Prodigy configuration: the SDXL-like workload's ten
    factored groups (2,602,705,920 params) attached to one controller (d0 1e-6, lr 1, beta2
    0.999, statistics on every 11th 64-element block, one gradient set reused), 5 steps.  The oracle steps every tensor
    (statistics before the update, the update with the step's d; tensors in parallel, sums in
    group and tensor order) and ends each step once; d after every step, every tensor's fp32
    master, p0 and s are checked with the tolerances of test_gpu_prodigy.py."""
    from test_gpu_prodigy import check, oracle_tensor
    cfg = W.config("sdxl_like")
    steps, slice_p, d0 = cfg["steps"], 11, 1e-6
    hp = dict(cfg["hp"], mode=1, lr=1.0, beta2=0.999, eps2=1e-30)
    ctrl = eng.ProdigyController(d0=d0, beta2=0.999, slice_p=slice_p)
    st = orc.ProdigyState(d0, ctrl.beta3, slice_p)
    groups, ora, tids, tid = [], [], [], 0
    for shapes in cfg["groups"]:
        ids = list(range(tid, tid + len(shapes)))
        masters = [W.master_weights(s, cfg["seed"], j, device="cuda") for s, j in zip(shapes, ids)]
        grp = eng.FactoredGroup.from_masters(masters)
        grp.attach_prodigy(ctrl)
        groups.append(grp)
        ora.append([oracle_tensor(orc, _f32(m), s, slice_p) for m, s in zip(masters, shapes)])
        del masters
        tids.append(ids)
        tid += len(shapes)

    def ora_tensor_step(tt, g, t, cs, d):
        dt, lt = orc.prodigy_tensor_stats(tt["hi"], tt["lo"], g, slice_p, tt["p0"], tt["s"], st.beta3, cs)
        orc.factored_group_step([tt], [g], t, dict(hp, d=d))
        return dt, lt

    ds, ds_ref, lrd = [], [], 0.0
    pool = ThreadPoolExecutor(max_workers=os.cpu_count() or 4)
    for t in range(1, steps + 1):
        d = st.d32
        lrd += hp["lr"] * d
        cdot, l1 = 0.0, 0.0
        for grp, shapes, ids, og in zip(groups, cfg["groups"], tids, ora):
            # one gradient set reused every step, as the benchmark does: the displacement then
            # correlates with the gradients and d grows
            grads = [W.grad_bf16(s, cfg["seed"], j, 1, cfg["g_std"], device="cuda") for s, j in zip(shapes, ids)]
            cr = float(np.float32(hp["lr"])) * d * d
            cs = float(np.float32(cr))
            futs = [pool.submit(ora_tensor_step, tt, _bits(g), t, cs, d) for tt, g in zip(og, grads)]
            grp.step(grads, hp)
            del grads
            dot_g = 0.0
            for f in futs:
                dt, lt = f.result()
                dot_g += dt
                l1 += lt
            cdot += cr * dot_g
        st.end_step(cdot, l1)
        ctrl.end_step()
        ds.append(ctrl.get()[0])
        ds_ref.append(st.d.value)
    pool.shutdown()
    torch.cuda.synchronize()
    assert ds_ref[-1] > d0                      # d moved during the run
    check(orc, ora, groups, ds, ds_ref, lrd)
    ctrl.close()
    torch.cuda.empty_cache()
