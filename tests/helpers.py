"""Shared helpers of the parity tests: build matching oracle / CUDA-path states from the same
seeded inputs and compare them.  Inputs come from memory_lean_optimizer_gb300.workloads; expected
values come only from the oracle."""
from __future__ import annotations

import numpy as np
import torch

from memory_lean_optimizer_gb300 import workloads as W

SMALL = 4096


def cuda_u16(a: np.ndarray) -> torch.Tensor:
    return W.from_bits16(a, "cuda")


def cuda_bits(t: torch.Tensor) -> np.ndarray:
    return W.bits16(t)


def alloc_offset(n: int, dtype, offset_elems: int, fill=0):
    """A contiguous CUDA buffer of n elements starting `offset_elems` past a 512-byte-aligned
    allocation (offset 1 gives a 2-byte aligned, not 16-byte aligned, pointer)."""
    base = torch.empty(n + offset_elems + 8, dtype=dtype, device="cuda")
    base.fill_(fill)
    return base, base[offset_elems:offset_elems + n]


class OracleNadam:
    """Oracle-side state of one NAdam group built from fp32 masters."""

    def __init__(self, orc, masters, kahan=True):
        self.orc = orc
        self.t = []
        for x in masters:
            x = np.ascontiguousarray(x, np.float32).reshape(-1)
            if kahan:
                hi, lo = orc.kahan_split(x)
            else:
                hi, lo = orc.round_bf16(x), None
            n = x.size
            if n <= SMALL:
                m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
            else:
                m, v = np.full(n, 32768, np.uint16), np.zeros(n, np.uint16)
            self.t.append(dict(hi=hi, lo=lo, m=m, v=v))
        self.state = orc.NadamState(len(self.t))
        self.step_count = 0

    def step(self, grads_u16, hp):
        self.step_count += 1
        self.orc.nadam_group_step(self.t, grads_u16, self.state, self.step_count, hp)

    def scales(self):
        return [self.state.scale(i) for i in range(len(self.t))]


def assert_nadam_equal(oracle: OracleNadam, group, tag=""):
    """Bit-exact comparison of weights, residuals and moment codes (or fp32 moments)."""
    for i, (ot, w) in enumerate(zip(oracle.t, group.weights)):
        n = ot["hi"].size
        if n == 0:
            continue
        hi = cuda_bits(w).reshape(-1)
        assert np.array_equal(hi, ot["hi"]), f"{tag} tensor {i} (n={n}): weight bits differ at {np.flatnonzero(hi != ot['hi'])[:5]}"
        if ot["lo"] is not None:
            lo = cuda_bits(group.res[i]).reshape(-1)
            assert np.array_equal(lo, ot["lo"]), f"{tag} tensor {i}: residual bits differ"
        if n <= SMALL:
            m = group.m[i].cpu().numpy()
            v = group.v[i].cpu().numpy()
            assert np.array_equal(m.view(np.uint32), ot["m"].view(np.uint32)), f"{tag} tensor {i}: fp32 m differs"
            assert np.array_equal(v.view(np.uint32), ot["v"].view(np.uint32)), f"{tag} tensor {i}: fp32 v differs"
        else:
            m = cuda_bits(group.m[i])
            v = cuda_bits(group.v[i])
            dm = np.abs(m.astype(np.int64) - ot["m"].astype(np.int64))
            dv = np.abs(v.astype(np.int64) - ot["v"].astype(np.int64))
            assert dm.max() == 0, f"{tag} tensor {i}: m codes differ (max {dm.max()}, count {(dm > 0).sum()})"
            assert dv.max() == 0, f"{tag} tensor {i}: v codes differ (max {dv.max()}, count {(dv > 0).sum()})"
