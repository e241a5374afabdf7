#!/usr/bin/env python
"""Throughput of the fused optimizer step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload flux19]

One step = one pass of the whole hot path over the workload: for the flux19 workload, the 19
group calls (one per Flux-like double-stream block, ~170M parameters each) of the fused
NAdamW + Kahan + u16-moment step, each a gradient-max pre-pass and the update kernel.  Inputs
(bf16 weights, residuals, moment codes, one set of bf16 gradients) are resident in HBM before
the timed region; together they are ~32 GB, far larger than L2, so no L2 flush is needed.

The JSON line reports params updated/s (whole job, all ranks), the step's HBM GB/s at the
algorithmic 18 bytes per parameter, a roofline record for the dominant kernel timed live with
CUDA events, the oracle's throughput on all host cores on a bounded sample, and an end-to-end
figure through the public API with the gradients copied in from pinned host memory and the
weights copied back every step.  The default run (flux19, one GPU) adds a `workloads` record with
the other workloads measured the same way, one after the other, each freed before the next: the
20,000-tensor ragged NAdam group, the SDXL-like factored step, the 35-group host-offload pipeline
and the single 1024x1024 tensor.  With N > 1 (torchrun), every rank steps its own copy of the
workload (weak scaling, no collective on the data path) and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "params updated/s and achieved HBM GB/s (% of GB300 roofline) per optimizer step"
BYTES_PER_PARAM_U16 = 18      # read w, res, g, m, v; write w, res, m, v (2 bytes each)
BYTES_PER_PARAM_F32 = 26      # fp32 moments: m, v 4 bytes each way
BYTES_PER_PARAM_F24 = 22      # f24 moments: m, v 3 bytes each way
PREPASS_BYTES_PER_PARAM = 2   # gradient-max pre-pass re-reads g
FALLBACK_HBM_GBS = 6800.0
# Source files of each measured kernel: a DRAM-traffic record is used only while they are unchanged.
KERNEL_SOURCES = {
    "k_nadam_step": ["memory_lean_optimizer_gb300/csrc/nadam.cu", "memory_lean_optimizer_gb300/csrc/common.cuh"],
    "k_nadam_step<sr>": ["memory_lean_optimizer_gb300/csrc/nadam.cu", "memory_lean_optimizer_gb300/csrc/common.cuh"],
    "k_nadam_f24": ["memory_lean_optimizer_gb300/csrc/nadam.cu", "memory_lean_optimizer_gb300/csrc/common.cuh"],
    "k_nadam_f24<sr>": ["memory_lean_optimizer_gb300/csrc/nadam.cu", "memory_lean_optimizer_gb300/csrc/common.cuh"],
    "k_adan_step": ["memory_lean_optimizer_gb300/csrc/adan.cu", "memory_lean_optimizer_gb300/csrc/common.cuh"],
    "k_adan_step<f24>": ["memory_lean_optimizer_gb300/csrc/adan.cu", "memory_lean_optimizer_gb300/csrc/common.cuh"],
    "factored_step": ["memory_lean_optimizer_gb300/csrc/factored.cu", "memory_lean_optimizer_gb300/csrc/common.cuh"],
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="flux19")
    p.add_argument("--states", default="u16", choices=["u16", "f24"],
                   help="state storage: NAdam u16 codes or f24; Adan fp32 (the default) or f24")
    p.add_argument("--optimizer", default="nadam", choices=["nadam", "adan", "prodigy"],
                   help="adan: fp32 m, v, n + previous gradient, Kahan residual (38 B/param); "
                        "prodigy (factored workloads): Prodigy mode with the step size d estimated each step")
    p.add_argument("--offload-slots", type=int, default=3, help="offload, engine form: device staging slots")
    p.add_argument("--offload-form", default="host", choices=["host", "engine"],
                   help="host: per-group calls (one pinned image per group, prefetch and write-back on the "
                        "caller's copy streams, library ring); engine: an engine object and per-state buffers")
    p.add_argument("--offload", action="store_true",
                   help="run the host-offload pipeline on this workload (flux35 always does); with "
                        "--optimizer adan the Adan states (fp32, or f24 with --states f24) are offloaded")
    p.add_argument("--slice-p", type=int, default=11, help="prodigy: statistics on every slice_p-th 64-element block")
    p.add_argument("--rounding", default="kahan", choices=["kahan", "sr"],
                   help="kahan: bf16 weight + u16 residual; sr: no residual, stochastic rounding")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-workloads", action="store_true", help="headline line only (no other workloads)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    return p.parse_args()


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if key in d and d[key]:
                    return float(d[key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_hash(kernel):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_per_launch(kernel, params_per_launch):
    """DRAM bytes per launch of `kernel` from the committed ncu record, scaled to the launch's
    parameter count (the kernels stream every parameter once, so traffic grows in proportion);
    None when absent or taken on different kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        e = d["kernels"].get(kernel)
        if e is None or e.get("kernel_source_sha") != kernel_hash(kernel):
            return None
        return e["dram_bytes_per_param"] * params_per_launch
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms; the summary keeps the samples
    taken inside the timed region (mark_start / mark_end bracket it), or all of them when the
    region is shorter than one sampling interval."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.2)      # the first sample before the timed region starts
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.t1 is None:
            self.mark_end()
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        from datetime import datetime

        def when(r):
            try:
                return datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except Exception:
                return None
        inside = [r for r in rows if when(r) is not None and self.t0 - 0.05 <= when(r) <= self.t1 + 0.05]
        use = inside if inside else rows
        sm = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in use if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


# ----------------------------------------------------------------------------- workload setup
def build_groups(cfg, device, rank, states="u16", rounding="kahan"):
    import torch
    from memory_lean_optimizer_gb300 import engine, workloads as W
    groups, grads, params = [], [], 0
    tid = 0
    for shapes in cfg["groups"]:
        masters, gs = [], []
        for s in shapes:
            masters.append(W.master_weights(s, cfg["seed"] + 1000 * rank, tid, device=device))
            gs.append(W.grad_bf16(s, cfg["seed"] + 1000 * rank, tid, 1, cfg["g_std"], device=device,
                                  zero_frac=cfg["zero_frac"]))
            params += W.numel(s)
            tid += 1
        if rounding == "sr":
            groups.append(engine.NadamGroup([x.to(torch.bfloat16) for x in masters], kahan=False, states=states))
        else:
            groups.append(engine.NadamGroup.from_masters(masters, states=states))
        del masters
        grads.append(gs)
    torch.cuda.synchronize()
    return groups, grads, params


def bytes_alg(shapes, states="u16", rounding="kahan"):
    from memory_lean_optimizer_gb300 import workloads as W
    tot = 0
    for s in shapes:
        n = W.numel(s)
        per = BYTES_PER_PARAM_F32 if n <= 4096 else (BYTES_PER_PARAM_F24 if states == "f24" else BYTES_PER_PARAM_U16)
        tot += n * (per - (4 if rounding == "sr" else 0))     # no residual read or written
    return tot


def _oracle_tensors(shapes, seed, first_tid, g_std, zero_frac):
    """Host copies of a list of tensors of the workload for the oracle: Kahan pair of the seeded
    fp32 masters, zero states, the step-1 bf16 gradients (the GPU arm's resident set)."""
    import numpy as np
    import oracle
    from memory_lean_optimizer_gb300 import workloads as W
    ts, gs = [], []
    for i, s in enumerate(shapes):
        x = W.master_weights(s, seed, first_tid + i).numpy().reshape(-1)
        hi, lo = oracle.kahan_split(x)
        n = x.size
        if n <= 4096:
            m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
        else:
            m, v = np.full(n, 32768, np.uint16), np.zeros(n, np.uint16)
        ts.append(dict(hi=hi, lo=lo, m=m, v=v))
        gs.append(W.bits16(W.grad_bf16(s, seed, first_tid + i, 1, g_std, zero_frac=zero_frac)).reshape(-1))
    return ts, gs


def cpu_baseline(cfg, target_s):
    """The oracle, as it stands, on every host core (its threaded timing driver: the same
    single-threaded step function over slices of the tensors, bit-identical results), on a bounded
    sample of the workload: its first groups, two steps each, until about target_s seconds of CPU
    time (wall time x threads) are spent."""
    import oracle
    oracle.build()
    cores = oracle.threads()
    done_params, wall, groups_done, tid = 0, 0.0, 0, 0
    for shapes in cfg["groups"]:
        if wall * cores >= target_s:
            break
        ts, gs = _oracle_tensors(shapes, cfg["seed"], tid, cfg["g_std"], cfg["zero_frac"])
        st = oracle.NadamState(len(ts))
        for step in (1, 2):
            t0 = time.perf_counter()
            oracle.nadam_group_step_mt(ts, gs, st, step, cfg["hp"])
            wall += time.perf_counter() - t0
            done_params += sum(t["hi"].size for t in ts)
        tid += len(shapes)
        groups_done += 1
        del ts, gs
    return {"value": done_params / wall, "unit": "params/s", "cores": cores, "kind": "oracle",
            "sample": f"the first {groups_done} groups of the workload ({done_params // 2} params) x 2 steps, "
                      f"{wall:.2f} s on {cores} threads ({wall * cores:.1f} thread-s)"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, cfg):
    """The oracle (threaded timing driver, every host core) stepping the whole workload: each step
    is every group call of the workload, as on the GPU, over the same tensors (inputs generated on
    the host with the same seeds and one resident gradient set).  Rank 0 only."""
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = oracle.threads()
    t_setup = time.perf_counter()
    groups, tid, params = [], 0, 0
    for shapes in cfg["groups"]:
        ts, gs = _oracle_tensors(shapes, cfg["seed"], tid, cfg["g_std"], cfg["zero_frac"])
        groups.append((ts, gs, oracle.NadamState(len(ts))))
        tid += len(shapes)
        params += sum(t["hi"].size for t in ts)
    t_setup = time.perf_counter() - t_setup
    step = 0

    def one_step():
        nonlocal step
        step += 1
        for ts, gs, st in groups:
            oracle.nadam_group_step_mt(ts, gs, st, step, cfg["hp"])

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = time.perf_counter() - t0
    value = params * args.steps / dt
    line = {"metric": METRIC, "value": value, "unit": "params/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(args, cfg, params, len(groups), world),
            "cpu_baseline": {"value": value, "unit": "params/s", "cores": cores, "kind": "oracle",
                             "sample": f"the whole workload ({params} params, {len(groups)} group calls) per step, "
                                       f"{cores} threads; setup {t_setup:.1f} s untimed"},
            "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(args, cfg, params, n_groups, world):
    """The `config` record of a NAdam workload line (shared by both arms)."""
    return {"workload": args.workload, "params_per_gpu": params, "groups": n_groups,
            "tensors": sum(len(s) for s in cfg["groups"]),
            "optimizer": f"NAdamW+{'Kahan' if args.rounding == 'kahan' else 'stochastic rounding'}, {args.states} moments",
            "lr": cfg["hp"]["lr"], "weight_decay": cfg["hp"]["weight_decay"],
            "grads": "one resident set reused each step",
            "l2": (f"inputs {params * 10 / 1e6:.1f} MB, inside the 129 MB L2: timed warm, reported only"
                   if params * 10 < 129e6 else
                   f"inputs ~{params * 10 / 1e9:.0f} GB per GPU, far above the 129 MB L2: no flush needed"),
            "parallelism": f"replicas x{world}"}


# ----------------------------------------------------------------------------- our arm
def run_ours(args, cfg):
    """The headline line: the NAdam workload (flux19 by default) with its e2e leg, then, on one GPU
    with the default workload, the other workloads as a `workloads` record, then the oracle
    baseline on the host."""
    import torch
    import torch.distributed as dist
    from memory_lean_optimizer_gb300 import build, lmopt, workloads as W

    world, rank, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    lmopt.load()
    result = measure_nadam(args, cfg, e2e=not args.no_e2e)
    torch.cuda.empty_cache()
    if world == 1 and args.workload == "flux19" and not args.no_workloads:
        result["workloads"] = other_workloads(args)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)
    return 0


def other_workloads(args):
    """The other workloads, each measured as its own bench line would be (same timing rules, live
    CUDA-event roofline of its dominant kernel, clocks sampled inside its timed region), each in a
    process of its own (so that no workload runs on the allocator state another one left), one
    after the other.  Returns name -> summary."""
    keep = ("ms_per_step", "value", "unit", "steps", "warmup", "roofline", "clocks", "ms_per_step_median",
            "first_step_ms", "hbm_gbs_step", "hbm_gbs_step_as_run", "link_gbs", "h2d_gbs", "d2h_gbs",
            "hbm_gbs_kernels_over_step", "link_peak_gbs", "link_probe_gbs", "step_ms", "gpu_launches", "config")
    plan = [("ragged20k", min(args.steps, 10)), ("sdxl_like", min(args.steps, 10)), ("flux35", 5), ("nadam_1m", 100)]
    out = {}
    for name, steps in plan:
        cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", name, "--steps", str(steps),
               "--warmup", str(max(3, args.warmup)), "--no-workloads", "--no-e2e", "--no-cpu-baseline"]
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
            lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
            if r.returncode != 0 or not lines:
                out[name] = {"error": f"exit {r.returncode}: {r.stderr.strip()[-300:]}"}
                continue
            d = json.loads(lines[-1])
            out[name] = {k: d[k] for k in keep if k in d}
        except Exception as e:            # one workload failing must not lose the headline line
            out[name] = {"error": f"{type(e).__name__}: {e}"[:400]}
    return out


def measure_nadam(args, cfg, e2e=True):
    """One NAdam workload (flux19, ragged20k, nadam_1m, ...): params/s, K2 roofline from live
    CUDA events, clocks; with e2e the public-API leg with host copies."""
    import torch
    import torch.distributed as dist
    from memory_lean_optimizer_gb300 import lmopt

    world, rank, local = dist_info()
    device = torch.device("cuda", local)

    groups, grads, params = build_groups(cfg, device, rank, args.states, args.rounding)
    hp = dict(cfg["hp"], stochastic_rounding=int(args.rounding == "sr"), seed=12345)
    stream = torch.cuda.current_stream()

    def one_step(events=None):
        for gi, (grp, gs) in enumerate(zip(groups, grads)):
            if events is not None:
                e0, em, e1 = events[gi]
                e0.record(stream)
                lmopt.optim_group_set_profile_event(grp.handle, em.cuda_event)
            grp.step(gs, hp, stream)
            if events is not None:
                e1.record(stream)
                lmopt.optim_group_set_profile_event(grp.handle, None)

    # the first step (t = 1: scales start from zero) timed on its own, then the other warm-ups
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for w in range(args.warmup):
        if w == 0:
            f0.record(stream)
        one_step()
        if w == 0:
            f1.record(stream)
    torch.cuda.synchronize()
    first_step_ms = f0.elapsed_time(f1) if args.warmup > 0 else None

    launches_per_step = sum(grp.launches(hp) for grp in groups)
    one_launch = all(grp.launches(hp) == 1 for grp in groups) and args.states == "u16"
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in groups] for _ in range(args.steps)]
    for per_step in ev:               # materialise the event handles the library records into
        for trio in per_step:
            for e in trio:
                e.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    start.record(stream)
    for k in range(args.steps):
        one_step(ev[k])
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    elapsed = start.elapsed_time(end) / 1e3
    if world > 1:
        t = torch.tensor([elapsed], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed = float(t.item())

    # per timed step: first group's start to last group's end
    step_ms = [ev[k][0][0].elapsed_time(ev[k][-1][2]) for k in range(args.steps)]
    # live per-kernel timing of the update kernel (between the library's mid event and the end)
    k2_ms, k1_ms = [], []
    for k in range(args.steps):
        for gi in range(len(groups)):
            e0, em, e1 = ev[k][gi]
            k1_ms.append(e0.elapsed_time(em))
            k2_ms.append(em.elapsed_time(e1))
    group_bytes = [bytes_alg(shapes, args.states, args.rounding) for shapes in cfg["groups"]]
    group_params = [sum(W_numel(s) for s in shapes) for shapes in cfg["groups"]]
    k2_bytes_total = sum(group_bytes) * args.steps
    k2_time_total = sum(k2_ms) / 1e3
    k2_gbs = k2_bytes_total / k2_time_total / 1e9
    peak, peak_src = peaks()
    params_per_launch = sum(group_params) / len(group_params)
    k2_name = ("k_nadam_f24" if args.states == "f24" else "k_nadam_fused" if one_launch else "k_nadam_step") + \
        ("<sr>" if args.rounding == "sr" else "")
    traffic = traffic_per_launch(k2_name, params_per_launch)

    step_s = elapsed / args.steps
    value = world * params * args.steps / elapsed
    result = {
        "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(args, cfg, params, len(groups), world),
        "hbm_gbs_step": sum(group_bytes) / step_s / 1e9,
        "hbm_gbs_step_as_run": (sum(group_bytes) + (PREPASS_BYTES_PER_PARAM * params if args.states == "u16" else 0)) / step_s / 1e9,
        "roofline": {"bound": "hbm", "kernel": k2_name,
                     "achieved": k2_gbs, "peak": peak, "unit": "GB/s",
                     "frac": k2_gbs / peak,
                     "traffic": traffic,
                     "peak_source": peak_src,
                     "bytes_per_param": (BYTES_PER_PARAM_F24 if args.states == "f24" else BYTES_PER_PARAM_U16)
                     - (4 if args.rounding == "sr" else 0),
                     "launch_ms_mean": 1e3 * k2_time_total / len(k2_ms),
                     "prepass_ms_mean": statistics.mean(k1_ms)},
        "gpu_launches": launches_per_step * args.steps,
        "ms_per_step_median": statistics.median(step_ms), "first_step_ms": first_step_ms,
        "clocks": clk,
    }

    if e2e:
        result["e2e"] = e2e_run(args, groups, grads, hp, params, stream, world, device)
    for grp in groups:
        grp.close()
    del groups, grads
    torch.cuda.empty_cache()
    return result


def e2e_run(args, groups, grads, hp, params, stream, world, device):
    """Same metric through the public API, host buffers: each step copies every group's bf16
    gradients from pinned host memory to the device, steps the group, and copies the updated bf16
    weights back to pinned host memory; all copies are inside the timed region.  Copies run on
    their own streams, ordered per group by events, so group k+1's copy-in and group k-1's
    copy-out overlap group k's kernels."""
    import torch
    import torch.distributed as dist
    host_g = [[g.to("cpu").pin_memory() for g in gs] for gs in grads]
    host_w = [[torch.empty(w.shape, dtype=w.dtype, pin_memory=True) for w in grp.weights] for grp in groups]
    steps = max(1, min(args.steps, 3))
    cin, cout = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    n = len(groups)
    done = [torch.cuda.Event() for _ in range(n)]      # group k's step finished (its buffers are free)
    for e in done:
        e.record(stream)

    def one():
        ins = []
        for k in range(n):
            cin.wait_event(done[k])                    # previous step no longer reads these gradients
            with torch.cuda.stream(cin):
                for d, h in zip(grads[k], host_g[k]):
                    d.copy_(h, non_blocking=True)
            e = torch.cuda.Event()
            e.record(cin)
            ins.append(e)
        for k in range(n):
            stream.wait_event(ins[k])
            groups[k].step(grads[k], hp, stream)
            done[k].record(stream)
            cout.wait_event(done[k])
            with torch.cuda.stream(cout):
                for h, w in zip(host_w[k], groups[k].weights):
                    h.copy_(w, non_blocking=True)

    # warm-up passes as for the device timing: the first passes over freshly pinned host buffers
    # run far below the link's rate (a bidirectional copy probe: 44 GB/s on its first repeat, 341
    # on the next), so one pass is not enough
    for _ in range(max(args.warmup, 1)):
        one()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    if world > 1:
        t = torch.tensor([dt], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dt = float(t.item())
    nbytes = 2 * params
    return {"value": world * params * steps / dt, "unit": "params/s", "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": nbytes, "steps": steps, "warmup": max(args.warmup, 1),
            "link_gbs": 2 * nbytes * steps / dt / 1e9}


def run_offload(args, cfg):
    import torch
    from memory_lean_optimizer_gb300 import build, lmopt
    torch.cuda.set_device(dist_info()[2])
    build.build()
    lmopt.load()
    print(json.dumps(measure_offload(args, cfg)), flush=True)
    return 0


def link_probe(device, nbytes=1 << 30, reps=3):
    """Pinned-host <-> device copy peak of this machine: both directions at once on two streams, best
    of `reps` after one warm-up repeat (GB/s, bytes both ways / time)."""
    import torch
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s1, s2 = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    best = 0.0
    for r in range(reps + 1):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        if r > 0:
            best = max(best, 2 * nbytes / dt / 1e9)
    del h_in, h_out, d_in, d_out
    return best


def measure_offload(args, cfg):
    """Host-offload workload (flux35): 35 Flux-like blocks, one group each, residuals and u16
    moments in pinned host memory (6 bytes per parameter), weights and gradients on the device.
    Each step prefetches group k+1 while group k updates and group k-1 writes back, through three
    staging slots: by default with the per-group calls (optim_group_attach_host: one pinned image per
    group, prefetch on a copy-in stream before each group's step, write-back on a copy-out stream
    after it), or with --offload-form engine through an engine object.  Reports params/s, the
    host-link GB/s both ways against a pinned copy probe on the same machine (taken before and after
    the timed steps, the better of the two as the peak: the host memory system may be shared), the
    time of each timed step, and the HBM GB/s of the update kernels."""
    import torch
    from memory_lean_optimizer_gb300 import engine, workloads as W
    world, rank, local = dist_info()
    device = torch.device("cuda", local)
    link_peak = link_probe(device)
    from memory_lean_optimizer_gb300 import lmopt
    adan = args.optimizer == "adan"
    kind = ((lmopt.OPTIM_KIND_ADAN_F24 if args.states == "f24" else lmopt.OPTIM_KIND_ADAN) if adan else
            (lmopt.OPTIM_KIND_NADAM_F24 if args.states == "f24" else lmopt.OPTIM_KIND_NADAM))
    shapes = cfg["groups"][0]
    slot = max(engine.offload_slot_bytes([W.numel(s) for s in g], kind=kind) for g in cfg["groups"])
    per_group = args.offload_form == "host"
    off = None if per_group else engine.OffloadEngine(slot, args.offload_slots)
    grads = [W.grad_bf16(s, cfg["seed"], i, 1, cfg["g_std"], device=device) for i, s in enumerate(shapes)]
    groups, params = [], 0
    t_setup = time.perf_counter()
    for gi, grp_shapes in enumerate(cfg["groups"]):
        masters = [W.master_weights(s, cfg["seed"], 1000 * gi + i, device=device) for i, s in enumerate(grp_shapes)]
        if adan:
            g = engine.AdanGroup.from_masters(masters, offload=off, states="f24" if args.states == "f24" else "fp32")
        else:
            g = engine.NadamGroup.from_masters(masters, offload=off, states=args.states)
        if per_group:
            g.attach_host()
        groups.append(g)
        params += sum(W.numel(s) for s in grp_shapes)
        del masters
    torch.cuda.synchronize()
    t_setup = time.perf_counter() - t_setup
    hp = ADAN_HP if adan else cfg["hp"]
    stream = torch.cuda.current_stream()

    cin, cout = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)

    def one_step():
        groups[0].prefetch(cin if per_group else None)
        for k, g in enumerate(groups):
            if k + 1 < len(groups):
                groups[k + 1].prefetch(cin if per_group else None)
            g.step(grads, hp, stream)
            if per_group:
                g.writeback(cout)

    def sync():
        torch.cuda.synchronize()
        return off.sync() if off is not None else engine.OffloadEngine.sync_library_ring()

    for _ in range(args.warmup):
        one_step()
    sync()
    b0 = sync()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    clocks = ClockSampler(local)
    clocks.start()
    t0 = time.perf_counter()
    marks[0].record(stream)
    for k in range(args.steps):
        one_step()
        marks[k + 1].record(stream)      # after the step's last update (its write-back may still run)
    b1 = sync()
    dt = time.perf_counter() - t0
    clk = clocks.stop()
    step_ms = [marks[k].elapsed_time(marks[k + 1]) for k in range(args.steps)]
    link_after = link_probe(device)      # a busy host memory system shows in this probe as well
    h2d = (b1[0] - b0[0]) / args.steps
    d2h = (b1[1] - b0[1]) / args.steps
    step_s = dt / args.steps
    hbm_bytes = params * (38 if adan and args.states != "f24" else 32 if adan else
                          BYTES_PER_PARAM_F24 if args.states == "f24" else BYTES_PER_PARAM_U16)
    link = (h2d + d2h) / step_s / 1e9
    peak = max(link_peak, link_after)
    result = {
        "metric": METRIC, "value": params * args.steps / dt, "unit": "params/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * step_s, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "params": params, "groups": len(groups),
                   "optimizer": ("Adan" if adan else "NAdam") + f" + Kahan, {args.states if (args.states == 'f24' or not adan) else 'fp32'} states",
                   "states": f"pinned host, {h2d / params:.0f} B/param each way",
                   "offload_form": ("per-group calls, one image per group, copy-in and copy-out streams"
                                    if per_group else f"engine, {args.offload_slots} staging slots"),
                   "staging_slots": 3 if per_group else args.offload_slots, "slot_bytes": slot, "setup_s": t_setup},
        "link_gbs": link, "h2d_gbs": h2d / step_s / 1e9, "d2h_gbs": d2h / step_s / 1e9,
        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "link_peak_gbs": peak,
        "link_probe_gbs": {"before": link_peak, "after": link_after}, "step_ms": step_ms,
        "roofline": {"bound": "host link", "kernel": "staging copies (both directions)", "achieved": link,
                     "peak": peak, "unit": "GB/s", "frac": link / peak if peak else None,
                     "traffic": None,
                     "peak_source": "measured: pinned copy probe, both directions at once, best of before and after"},
        "hbm_gbs_kernels_over_step": hbm_bytes / step_s / 1e9,
        "gpu_launches": (1 if adan or args.states == "f24" else 2) * len(groups) * args.steps,
        "clocks": clk,
    }
    for g in groups:
        g.close()
    if off is not None:
        off.close()
    return result


ADAN_HP = dict(lr=3.3e-5, beta1=0.02, beta2=0.08, beta3=0.01, eps=1e-8, weight_decay=0.02)


def run_adan(args, cfg):
    """Adan over the NAdam workload's tensors (flux19 by default): one kernel per group call."""
    import torch
    from memory_lean_optimizer_gb300 import build, engine, lmopt, workloads as W
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    build.build()
    lmopt.load()
    groups, grads, params, tid = [], [], 0, 0
    for shapes in cfg["groups"]:
        masters = [W.master_weights(s, cfg["seed"], tid + i, device=device) for i, s in enumerate(shapes)]
        grads.append([W.grad_bf16(s, cfg["seed"], tid + i, 1, cfg["g_std"], device=device) for i, s in enumerate(shapes)])
        groups.append(engine.AdanGroup.from_masters(masters, states="f24" if args.states == "f24" else "fp32"))
        params += sum(W.numel(s) for s in shapes)
        tid += len(shapes)
        del masters
    hp = ADAN_HP
    bpp = 32 if args.states == "f24" else 38
    stream = torch.cuda.current_stream()

    def one_step():
        for g, gs in zip(groups, grads):
            g.step(gs, hp, stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    start.record(stream)
    for _ in range(args.steps):
        one_step()
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    step_s = start.elapsed_time(end) / 1e3 / args.steps
    peak, src = peaks()
    gbs = bpp * params / step_s / 1e9
    print(json.dumps({
        "metric": METRIC, "value": params / step_s, "unit": "params/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "params": params,
                   "optimizer": f"Adan + Kahan, {'f24' if bpp == 32 else 'fp32'} m/v/n + previous bf16 grad"},
        "roofline": {"bound": "hbm", "kernel": "k_adan_step" + ("<f24>" if bpp == 32 else ""), "achieved": gbs,
                     "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": traffic_per_launch("k_adan_step" + ("<f24>" if bpp == 32 else ""), params / len(groups)),
                     "peak_source": src, "bytes_per_param": bpp},
        "gpu_launches": len(groups) * args.steps, "clocks": clk}), flush=True)
    for g in groups:
        g.close()
    return 0


def factored_bytes(shape):
    """Algorithmic HBM bytes of one factored step of a tensor: g read once (2 B/elem), weight and
    residual read and written (8 B/elem), fp32 statistics read and written."""
    n = W_numel(shape)
    if len(shape) >= 2:
        lead = W_numel(shape[:-2]) if len(shape) > 2 else 1
        state = lead * (shape[-2] + shape[-1])
    else:
        state = n
    return 10 * n + 8 * state


def prodigy_bytes(shape, slice_p):
    """Algorithmic HBM bytes of one tensor's Prodigy statistics: p0 read, s read and written
    (12 B per sampled element; the sampled weights and gradients are counted once, by the
    factored step)."""
    blocks = (W_numel(shape) + 63) // 64
    return 12 * 64 * ((blocks + slice_p - 1) // slice_p)


def run_factored(args, cfg):
    import torch
    import torch.distributed as dist
    from memory_lean_optimizer_gb300 import build, lmopt
    world, rank, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    lmopt.load()
    result = measure_factored(args, cfg)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)
    return 0


def measure_factored(args, cfg):
    """Factored workload (sdxl_like): Adafactor mode over 1332 SDXL-UNet-like tensors in 10
    groups, every step all group calls; reports params/s and HBM GB/s at the algorithmic bytes.
    --optimizer prodigy: Prodigy mode (lr 1, beta2 0.999) with every group attached to one
    controller, each step all group calls and the controller's end of step."""
    import torch
    import torch.distributed as dist
    from memory_lean_optimizer_gb300 import engine, workloads as W
    world, rank, local = dist_info()
    device = torch.device("cuda", local)
    groups, grads, params, nbytes, tid = [], [], 0, 0, 0
    for shapes in cfg["groups"]:
        masters = [W.master_weights(s, cfg["seed"], tid + i, device=device) for i, s in enumerate(shapes)]
        grads.append([W.grad_bf16(s, cfg["seed"], tid + i, 1, cfg["g_std"], device=device) for i, s in enumerate(shapes)])
        groups.append(engine.FactoredGroup.from_masters(masters))
        params += sum(W.numel(s) for s in shapes)
        nbytes += sum(factored_bytes(s) for s in shapes)
        tid += len(shapes)
        del masters
    hp = cfg["hp"]
    stream = torch.cuda.current_stream()
    ctrl = None
    if args.optimizer == "prodigy":
        hp = dict(hp, mode=1, lr=1.0, beta2=0.999, eps2=1e-30)
        ctrl = engine.ProdigyController(d0=1e-6, beta2=0.999, slice_p=args.slice_p)
        for g in groups:
            g.attach_prodigy(ctrl, stream)
        nbytes += sum(prodigy_bytes(s, args.slice_p) for shapes in cfg["groups"] for s in shapes)

    def one_step():
        for g, gs in zip(groups, grads):
            g.step(gs, hp, stream)
        if ctrl is not None:
            ctrl.end_step(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    start.record(stream)
    for _ in range(args.steps):
        one_step()
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_s = start.elapsed_time(end) / 1e3 / args.steps
    if world > 1:                     # one replica per rank (weak scaling): the slowest rank
        t = torch.tensor([step_s], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_s = float(t.item())
    peak, src = peaks()
    gbs = nbytes / step_s / 1e9
    result = {
        "metric": METRIC, "value": world * params / step_s, "unit": "params/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "params": params, "groups": len(groups),
                   "optimizer": ("Adafactor factored v, beta1=0, Kahan, clip 1.0" if ctrl is None else
                                 f"Prodigy factored v, beta1=0, d estimated each step (slice_p {args.slice_p}), "
                                 "Kahan, clip 1.0"),
                   "bytes_per_step_algorithmic": nbytes, "parallelism": f"replicas x{world}",
                   "l2": "inputs ~26 GB, far above the 129 MB L2: no flush needed"},
        "roofline": {"bound": "hbm", "kernel": "factored step (stats+final+rms+apply)", "achieved": gbs,
                     "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     # per step (the roofline object covers the whole step): the Adafactor step's
                     # DRAM bytes per parameter from a warm-L2 capture, scaled to this step
                     "traffic": traffic_per_launch("factored_step", params) if ctrl is None else None,
                     "peak_source": src},
        "clocks": clk,
    }
    if ctrl is not None:
        result["prodigy_d"] = ctrl.get()[0]
        ctrl.close()
    for g in groups:
        g.close()
    return result


def W_numel(shape):
    n = 1
    for s in shape:
        n *= int(s)
    return n


def main():
    args = parse()
    from memory_lean_optimizer_gb300 import workloads as W
    cfg = W.config(args.workload)
    if args.impl == "reference":
        if cfg["kind"] != "nadam" or args.optimizer != "nadam" or args.states != "u16":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the NAdam u16 oracle; "
                              "other optimizers and storages are GPU-only lines"}), flush=True)
            return 0
        return run_reference(args, cfg)
    if args.workload == "flux35" or args.offload:
        return run_offload(args, cfg)
    if cfg["kind"] == "factored":
        return run_factored(args, cfg)
    if args.optimizer == "adan":
        return run_adan(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
