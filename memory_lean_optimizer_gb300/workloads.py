"""Seeded synthetic workloads: tensor shapes and input generators.

This module holds no optimizer arithmetic: only shapes, random draws and dtype casts.  Both the
CUDA path and the CPU oracle consume what it produces.  Inputs are drawn with torch generators
(on the CPU for parity tests, on the GPU for full-size runs); each tensor gets its own seed
derived from (seed, tensor index, step, stream id), so any tensor can be regenerated alone.

Workloads (shapes stand in for Flux and SDXL weights, which are not needed: all inputs are
synthetic):
  nadam_1m     one 1024x1024 bf16 weight, 10 steps
  flux19       19 Flux-like double-stream blocks x {3072x9216, 3072x3072, 3072x12288,
               12288x3072, 3072x18432}: 3,227,516,928 parameters, one group per block
  sdxl_like    SDXL-UNet-like linears, 3x3 convs and 1-D tensors, 2,602,705,920 parameters,
               10 groups
  ragged20k    20,000 tensors, sizes round(2^U(6,22)), 1% exact-zero gradients
  flux35       35 Flux-like blocks (5,945,425,920 parameters) for the host-offload pipeline
"""
from __future__ import annotations

import math

import numpy as np
import torch

FLUX_BLOCK = [(3072, 9216), (3072, 3072), (3072, 12288), (12288, 3072), (3072, 18432)]

W_STD = 0.02


def flux_shapes(blocks: int = 19):
    """Per block, the five Flux-like double-stream linear shapes."""
    return [list(FLUX_BLOCK) for _ in range(blocks)]


def ragged_sizes(n: int = 20000, seed: int = 0, lo_exp: float = 6.0, hi_exp: float = 22.0):
    """n sizes round(2^U(lo_exp, hi_exp)), seeded."""
    rng = np.random.default_rng(seed)
    return [int(round(2.0 ** e)) for e in rng.uniform(lo_exp, hi_exp, n)]


def sdxl_like_shapes():
    """SDXL-UNet-like tensor list: 60 transformer(1280) + 12 transformer(640) blocks, where
    transformer(c) = 6x(c,c), 2x(c,2048), (8c,c), (c,4c), 6x(c,); 3x3 convs (c,c,3,3) x
    {1280: 20, 640: 24, 320: 16}, each with 2 bias vectors.  1332 tensors, 2,602,705,920 params."""
    shapes = []
    for c, reps in ((1280, 60), (640, 12)):
        for _ in range(reps):
            shapes += [(c, c)] * 6 + [(c, 2048)] * 2 + [(8 * c, c), (c, 4 * c)] + [(c,)] * 6
    for c, reps in ((1280, 20), (640, 24), (320, 16)):
        for _ in range(reps):
            shapes += [(c, c, 3, 3), (c,), (c,)]
    return shapes


def numel(shape) -> int:
    return int(math.prod(shape))


def balanced_groups(shapes, n_groups: int):
    """Contiguous split of a tensor list into n_groups groups of roughly equal element count."""
    n_groups = max(1, min(n_groups, len(shapes)))
    total = sum(numel(s) for s in shapes)
    groups, cur, acc = [], [], 0
    for i, s in enumerate(shapes):
        cur.append(s)
        acc += numel(s)
        left_groups, left_shapes = n_groups - len(groups) - 1, len(shapes) - i - 1
        if left_groups > 0 and (acc >= total * (len(groups) + 1) / n_groups or left_shapes == left_groups):
            groups.append(cur)
            cur = []
    if cur:
        groups.append(cur)
    return groups


def _gen(seed: int, tensor: int, step: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tensor * 7919 + step * 104_729 + stream * 15_485_863) % (2 ** 63))
    return g


def master_weights(shape, seed: int, tensor: int, device="cpu", std: float = W_STD) -> torch.Tensor:
    """fp32 master weights ~ N(0, std)."""
    g = _gen(seed, tensor, 0, 1, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(std)


def grad_bf16(shape, seed: int, tensor: int, step: int, std: float, device="cpu",
              zero_frac: float = 0.0) -> torch.Tensor:
    """bf16 gradient ~ N(0, std) (round-to-nearest cast), with i.i.d. exact zeros at zero_frac."""
    g = _gen(seed, tensor, step, 2, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(std)
    if zero_frac > 0:
        x.masked_fill_(torch.rand(shape, generator=g, device=device) < zero_frac, 0.0)
    return x.to(torch.bfloat16)


def bits16(t: torch.Tensor) -> np.ndarray:
    """Host uint16 view of a 16-bit tensor (bf16 or int16)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits16(a: np.ndarray, device="cpu") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)


# configuration records: name -> dict(kind, shapes per group, hyper-parameters, steps, std)
NADAM_HP = dict(lr=3.5e-6, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, wd_mode=0, nesterov=1,
                momentum_decay=0.004)


def config(name: str):
    if name == "nadam_1m":
        return dict(kind="nadam", groups=[[(1024, 1024)]], hp=dict(NADAM_HP), steps=10, g_std=1e-3,
                    zero_frac=0.0, seed=0)
    if name == "flux19":
        return dict(kind="nadam", groups=flux_shapes(19), hp=dict(NADAM_HP, weight_decay=0.01, wd_mode=1),
                    steps=5, g_std=1e-4, zero_frac=0.0, seed=0)
    if name == "flux1":   # one block (~170M parameters, ~1.7 GB resident): the profiling case
        return dict(kind="nadam", groups=flux_shapes(1), hp=dict(NADAM_HP, weight_decay=0.01, wd_mode=1),
                    steps=5, g_std=1e-4, zero_frac=0.0, seed=0)
    if name == "ragged20k":
        return dict(kind="nadam", groups=[[(n,) for n in ragged_sizes(20000, 0)]], hp=dict(NADAM_HP),
                    steps=5, g_std=1e-3, zero_frac=0.01, seed=0)
    if name == "ragged1k":   # the first 1,000 tensors of ragged20k (~0.4e9 parameters): its profiling case
        c = config("ragged20k")
        c["groups"] = [c["groups"][0][:1000]]
        return c
    if name == "sdxl_like":
        # ten optimizer groups: the group count the SDXL optimizer-groups option recommends (4-10)
        shapes = sdxl_like_shapes()
        return dict(kind="factored", groups=balanced_groups(shapes, 10),
                    hp=dict(lr=2e-6, beta2=0.999, decay_rate=-0.8, eps1=1e-30, eps2=1e-30, d=1.0,
                            clip_threshold=1.0, weight_decay=0.0, mode=0),
                    steps=5, g_std=1e-4, zero_frac=0.0, seed=0)
    if name == "sdxl_like_1":   # the first group of sdxl_like (~260M parameters): the profiling case
        c = config("sdxl_like")
        c["groups"] = c["groups"][:1]
        return c
    if name == "sdxl_like_conv":   # the 3x3 convolutions of sdxl_like, one group: small-matrix profiling
        c = config("sdxl_like")
        c["groups"] = [[s for s in sdxl_like_shapes() if len(s) == 4]]
        return c
    if name == "flux35":
        return dict(kind="nadam", groups=flux_shapes(35), hp=dict(NADAM_HP), steps=3, g_std=1e-4,
                    zero_frac=0.0, seed=0)
    raise KeyError(name)
