"""Parity at full workload sizes, in the launch configuration the benchmark times (one library
group per Flux-like block, the ten SDXL-like factored groups, one group of 20,000 ragged tensors, the
35-group host-offload pipeline).  The oracle replays whole sampled tensors -- their inputs are
copied back from the device before each step -- and the remaining tensors are checked through
properties that hold at any size (finite results, scale records bounding their maxima)."""
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


def _check_nadam_tensor(ora, i_ora, grp, i_grp, tag):
    ot = ora.t[i_ora]
    assert np.array_equal(_bits(grp.weights[i_grp]), ot["hi"]), f"{tag}: weights differ"
    assert np.array_equal(_bits(grp.res[i_grp]), ot["lo"]), f"{tag}: residuals differ"
    if ot["hi"].size > 4096:
        assert np.array_equal(_bits(grp.m[i_grp]), ot["m"]), f"{tag}: m codes differ"
        assert np.array_equal(_bits(grp.v[i_grp]), ot["v"]), f"{tag}: v codes differ"
    else:
        assert np.array_equal(grp.m[i_grp].cpu().numpy().reshape(-1), ot["m"])
        assert np.array_equal(grp.v[i_grp].cpu().numpy().reshape(-1), ot["v"])


def _scale_records_bound(grp, n):
    from memory_lean_optimizer_gb300 import lmopt
    recs = lmopt.optim_query_scales(grp.handle, n)
    for s_m, s_v, a_m, a_v in recs:
        assert np.isfinite([s_m, s_v, a_m, a_v]).all()
        assert a_m <= s_m * (1 + 1e-4) + 1e-30 and a_v <= s_v * (1 + 1e-4) + 1e-30
    assert lmopt.optim_query_nonfinite(grp.handle) == 0


def test_flux19_full(orc, eng):
    """19 blocks x 5 Flux-like linears (3,227,516,928 params), NAdamW wd 0.01, 2 steps; block 0
    and the last block's largest tensor replayed whole by the oracle."""
    cfg = W.config("flux19")
    hp, steps = cfg["hp"], 2
    sample = {(0, i) for i in range(5)} | {(18, 4)}
    groups, shapes_all, ora = [], [], {}
    tid = 0
    for b, shapes in enumerate(cfg["groups"]):
        masters = []
        for i, s in enumerate(shapes):
            x = W.master_weights(s, 0, tid, device="cuda")
            if (b, i) in sample:
                ora[(b, i)] = OracleNadam(orc, [x.cpu().numpy()])
            masters.append(x)
            tid += 1
        groups.append(eng.NadamGroup.from_masters(masters))
        shapes_all.append(shapes)
        del masters
    for t in range(1, steps + 1):
        tid = 0
        for b, (grp, shapes) in enumerate(zip(groups, shapes_all)):
            grads = []
            for i, s in enumerate(shapes):
                g = W.grad_bf16(s, 0, tid, t, cfg["g_std"], device="cuda")
                if (b, i) in sample:
                    ora[(b, i)].step([_bits(g)], hp)
                grads.append(g)
                tid += 1
            grp.step(grads, hp)
            del grads
    torch.cuda.synchronize()
    for (b, i), o in ora.items():
        _check_nadam_tensor(o, 0, groups[b], i, f"block {b} tensor {i}")
    for grp in groups:
        _scale_records_bound(grp, 5)
        grp.close()
    del groups
    torch.cuda.empty_cache()


def test_ragged20k_full(orc, eng):
    """20,000 tensors (sizes round(2^U(6,22)), ~7.56e9 params, 37.5% with fp32 moments), 1%
    exact-zero gradients, one group, 2 steps; 40 tensors replayed whole, including the largest
    and several of 4096 or fewer elements."""
    cfg = W.config("ragged20k")
    hp, steps = cfg["hp"], 2
    sizes = [s[0] for s in cfg["groups"][0]]
    rng = np.random.default_rng(0)
    sample = set(rng.choice(len(sizes), 36, replace=False).tolist()) | {int(np.argmax(sizes)), int(np.argmin(sizes))}
    sample |= {i for i, n in enumerate(sizes) if n in (4096, 4097)}
    sample = sorted(sample)[:40]
    masters = [W.master_weights((n,), 0, i, device="cuda") for i, n in enumerate(sizes)]
    ora = OracleNadam(orc, [masters[i].cpu().numpy() for i in sample])
    grp = eng.NadamGroup.from_masters(masters)
    del masters
    for t in range(1, steps + 1):
        grads = [W.grad_bf16((n,), 0, i, t, cfg["g_std"], device="cuda", zero_frac=0.01) for i, n in enumerate(sizes)]
        ora.step([_bits(grads[i]) for i in sample], hp)
        grp.step(grads, hp)
        del grads
    torch.cuda.synchronize()
    for j, i in enumerate(sample):
        _check_nadam_tensor(ora, j, grp, i, f"tensor {i} (n={sizes[i]})")
    _scale_records_bound(grp, len(sizes))
    grp.close()
    del grp
    torch.cuda.empty_cache()


def test_sdxl_like_full(orc, eng):
    """SDXL-like factored workload (1332 tensors, 2,602,705,920 params) in its 10 groups,
    Adafactor mode, 2 steps; one linear of each kind, a 3x3 conv and 1-D tensors replayed whole."""
    from test_gpu_factored import OracleFactored
    cfg = W.config("sdxl_like")
    hp, steps = cfg["hp"], 2
    shapes = [s for g in cfg["groups"] for s in g]
    want = {(10240, 1280), (1280, 5120), (640, 640), (1280, 1280, 3, 3), (320, 320, 3, 3), (1280,), (320,)}
    sample, seen = [], set()
    for i, s in enumerate(shapes):
        if tuple(s) in want and tuple(s) not in seen:
            sample.append(i)
            seen.add(tuple(s))
    masters = [W.master_weights(s, 0, i, device="cuda") for i, s in enumerate(shapes)]
    ora = OracleFactored(orc, [masters[i].cpu().numpy() for i in sample], [shapes[i] for i in sample])
    bounds = np.cumsum([0] + [len(g) for g in cfg["groups"]])
    groups = [eng.FactoredGroup.from_masters(masters[bounds[k]:bounds[k + 1]]) for k in range(len(cfg["groups"]))]
    del masters
    for t in range(1, steps + 1):
        grads = [W.grad_bf16(s, 0, i, t, cfg["g_std"], device="cuda") for i, s in enumerate(shapes)]
        ora.step([_bits(grads[i]) for i in sample], hp)
        for k, grp in enumerate(groups):
            grp.step(grads[bounds[k]:bounds[k + 1]], hp)
        del grads
    torch.cuda.synchronize()
    for j, i in enumerate(sample):
        k = int(np.searchsorted(bounds, i, side="right")) - 1
        grp, li = groups[k], i - int(bounds[k])
        ot = ora.t[j]
        ref = orc.kahan_merge(ot["hi"], ot["lo"]).astype(np.float64)
        got = grp.masters()[li].cpu().numpy().reshape(-1).astype(np.float64)
        tol = 1e-6 * np.abs(ref) + 1e-6 * hp["lr"] * steps
        assert np.all(np.abs(got - ref) <= tol), f"tensor {i} {shapes[i]}: masters differ"
        if "row" in ot:
            for name, st in (("row", grp.row[li]), ("col", grp.col[li])):
                r = ot[name].astype(np.float64)
                assert np.all(np.abs(st.cpu().numpy() - r) <= 2e-6 * np.abs(r) + 1e-37)
    for grp in groups:
        for w in grp.masters():
            assert torch.isfinite(w).all()
        grp.close()
    del groups
    torch.cuda.empty_cache()


def test_flux35_offload_full(orc, eng):
    """35 Flux-like blocks (5,945,425,920 params) with residuals and u16 moments in pinned host
    memory (35.7 GB), 3 staging slots, 2 steps; block 0 and block 34 replayed whole."""
    cfg = W.config("flux35")
    hp, steps = cfg["hp"], 2
    shapes = cfg["groups"][0]
    slot = eng.offload_slot_bytes([W.numel(s) for s in shapes])
    off = eng.OffloadEngine(slot, 3)
    sample_blocks = (0, 34)
    groups, ora = [], {}
    for b in range(35):
        masters = [W.master_weights(s, 0, 1000 * b + i, device="cuda") for i, s in enumerate(shapes)]
        if b in sample_blocks:
            ora[b] = OracleNadam(orc, [x.cpu().numpy() for x in masters])
        groups.append(eng.NadamGroup.from_masters(masters, offload=off))
        del masters
    for t in range(1, steps + 1):
        grads = [W.grad_bf16(s, 0, i, t, cfg["g_std"], device="cuda") for i, s in enumerate(shapes)]
        gb = [_bits(g) for g in grads]
        for b in sample_blocks:
            ora[b].step(gb, hp)
        groups[0].prefetch()
        for k, grp in enumerate(groups):
            if k + 1 < len(groups):
                groups[k + 1].prefetch()
            grp.step(grads, hp)
        del grads
    off.sync()
    torch.cuda.synchronize()
    for b in sample_blocks:
        for i in range(len(shapes)):
            ot = ora[b].t[i]
            g = groups[b]
            assert np.array_equal(_bits(g.weights[i]), ot["hi"])
            assert np.array_equal(g.res[i].numpy().view(np.uint16).reshape(-1), ot["lo"])
            assert np.array_equal(g.m[i].numpy().view(np.uint16).reshape(-1), ot["m"])
            assert np.array_equal(g.v[i].numpy().view(np.uint16).reshape(-1), ot["v"])
    for g in groups:
        g.close()
    off.close()
    del groups
    torch.cuda.empty_cache()


def test_tensor_beyond_2_31_elements(orc, eng):
    """One tensor of 2^31 + 13 elements (64-bit element offsets, 131,073 chunks), one NAdamW
    step: sampled elements -- chunk edges, both sides of 2^31, the last one, random ones -- equal
    the oracle's step of the same element, given the tensor's max|g| computed on the host."""
    n = (1 << 31) + 13
    hp = dict(W.NADAM_HP, weight_decay=0.01, wd_mode=1)
    master = W.master_weights((n,), 3, 0, device="cuda")
    grp = eng.NadamGroup.from_masters([master])
    rng = np.random.default_rng(0)
    idx = np.unique(np.concatenate([[0, 1, 7, 8, 16383, 16384, (1 << 31) - 1, 1 << 31, (1 << 31) + 5, n - 1],
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
