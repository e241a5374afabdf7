"""Torch-facing parameter groups over liblmopt.so.

PyTorch provides device memory and streams only: every step, split, merge, pack and unpack is a
library kernel called through the C ABI (``lmopt``).  A group owns the optimizer state of its
tensors (Kahan residuals, moments or factored statistics) as torch tensors, registers them once
with ``optim_group_create`` and then steps them with one library call per group -- the
granularity of the fused backward pass and of optimizer groups ("Fused backward pass" commit,
README: per-parameter hook, optimizer groups of 4-10).
"""
from __future__ import annotations

from typing import Sequence

import torch

from . import lmopt

SMALL = lmopt.SMALL_NUMEL


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _u16_empty(n: int, device, fill: int | None = None) -> torch.Tensor:
    """A uint16 buffer held as int16 storage (bit pattern only)."""
    t = torch.empty(n, dtype=torch.int16, device=device)
    if fill is not None:
        t.fill_(fill - 65536 if fill >= 32768 else fill)
    return t


def kahan_split(master: torch.Tensor, hi: torch.Tensor | None = None, lo: torch.Tensor | None = None, stream=None):
    """fp32 master -> (bf16 weight, int16-stored residual) via the library kernel."""
    assert master.dtype == torch.float32 and master.is_cuda and master.is_contiguous()
    if hi is None:
        hi = torch.empty(master.shape, dtype=torch.bfloat16, device=master.device)
    if lo is None:
        lo = _u16_empty(master.numel(), master.device)
    lmopt.optim_kahan_split(master.data_ptr(), hi.data_ptr(), lo.data_ptr(), master.numel(), _stream_ptr(stream))
    return hi, lo


def kahan_merge(hi: torch.Tensor, lo: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    if out is None:
        out = torch.empty(hi.shape, dtype=torch.float32, device=hi.device)
    lmopt.optim_kahan_merge(hi.data_ptr(), lo.data_ptr(), out.data_ptr(), hi.numel(), _stream_ptr(stream))
    return out


def state_pack(x: torch.Tensor, is_signed: bool, stream=None):
    codes = _u16_empty(x.numel(), x.device)
    scale = torch.empty(1, dtype=torch.float32, device=x.device)
    lmopt.state_pack_u16(x.data_ptr(), codes.data_ptr(), scale.data_ptr(), x.numel(), is_signed, _stream_ptr(stream))
    return codes, scale


def state_unpack(codes: torch.Tensor, scale: torch.Tensor, is_signed: bool, stream=None):
    out = torch.empty(codes.numel(), dtype=torch.float32, device=codes.device)
    lmopt.state_unpack_u16(codes.data_ptr(), scale.data_ptr(), out.data_ptr(), codes.numel(), is_signed,
                           _stream_ptr(stream))
    return out


def _desc(w, res, m, v, shape) -> lmopt.TensorDesc:
    d = lmopt.TensorDesc()
    d.w_bf16 = w.data_ptr() if w.numel() else None
    d.res_u16 = res.data_ptr() if (res is not None and res.numel()) else None
    d.m = m.data_ptr() if (m is not None and m.numel()) else None
    d.v = v.data_ptr() if (v is not None and v.numel()) else None
    d.numel = w.numel()
    shape = tuple(shape) if len(shape) else (w.numel(),)
    d.ndim = len(shape)
    for i, s in enumerate(shape):
        d.shape[i] = int(s)
    return d


class _Group:
    kind = -1

    def __init__(self):
        self.handle = None
        self.step_count = 0

    def close(self):
        if self.handle:
            lmopt.optim_group_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # attribute names of the (residual, m, v) state lists, in the order of optim_offload_layout
    _state_attrs = ("res", "m", "v")

    def attach_host(self):
        """Moves the group's residuals and states into one pinned host image (optim_group_attach_host);
        afterwards each step needs prefetch() before and writeback() after it, and the state lists
        of this object are views into the image (valid once the write-back has completed)."""
        total, offs = lmopt.optim_offload_layout(self.handle, len(self.weights))
        image = torch.zeros(max(total, 1), dtype=torch.uint8, pin_memory=True)
        lmopt.optim_group_attach_host(self.handle, image.data_ptr(), total)
        self.image = image
        for k, name in enumerate(self._state_attrs):
            views = []
            for i, t in enumerate(getattr(self, name)):
                if t is None or offs[i][k] < 0:
                    views.append(t if t is None else t.cpu())
                    continue
                nbytes = t.numel() * t.element_size()
                views.append(image[offs[i][k]:offs[i][k] + nbytes].view(t.dtype).view(t.shape))
            setattr(self, name, views)     # the device buffers are no longer used: dropped here

    def prefetch(self, stream=None):
        """Copy-in of an offloaded group's states (stream None: the library's own copy stream)."""
        lmopt.optim_offload_prefetch(self.handle, 0 if stream is None else int(stream.cuda_stream))

    def writeback(self, stream=None):
        """Copy-out after the last step of a group attached with attach_host()."""
        lmopt.optim_offload_writeback(self.handle, 0 if stream is None else int(stream.cuda_stream))

    def _grad_ptrs(self, grads):
        assert len(grads) == len(self.weights)
        ptrs = []
        for g, w in zip(grads, self.weights):
            assert g.dtype == torch.bfloat16 and g.is_contiguous() and g.numel() == w.numel()
            ptrs.append(g.data_ptr() if g.numel() else None)
        return ptrs


def _round256(x: int) -> int:
    return (x + 255) & ~255


def offload_slot_bytes(numels: Sequence[int], kahan: bool = True, kind: int = lmopt.OPTIM_KIND_NADAM) -> int:
    """Staging bytes one offloaded group of tensors with these sizes needs in a slot (the layout
    of optim_offload_layout: residual, m, v per tensor, each at a 256-byte boundary)."""
    tot = 0
    for n in numels:
        if n == 0:
            continue
        small = n <= SMALL
        f24 = (2 * n + 15) // 16 * 16 + n
        if kind == lmopt.OPTIM_KIND_NADAM:
            m = v = (4 if small else 2) * n
        elif kind == lmopt.OPTIM_KIND_NADAM_F24:
            m = v = 4 * n if small else f24
        else:
            m = 12 * ((n + 3) // 4 * 4) if (small or kind == lmopt.OPTIM_KIND_ADAN) else 3 * adan_f24_stride(n)
            v = 2 * n
        tot += (_round256(2 * n) if kahan else 0) + _round256(m) + _round256(v)
    return tot


class OffloadEngine:
    """Device staging ring + copy streams for groups whose states live in pinned host memory
    (None: the library's own ring of the current device, used by attach_host groups)."""

    def __init__(self, slot_bytes: int, n_slots: int = 3):
        self.handle = lmopt.optim_offload_create(int(slot_bytes), int(n_slots))

    def sync(self):
        return lmopt.optim_offload_sync(self.handle)

    @staticmethod
    def sync_library_ring():
        return lmopt.optim_offload_sync(None)

    def close(self):
        if self.handle:
            lmopt.optim_offload_destroy(self.handle)
            self.handle = None


def _state_buffer(n: int, dtype, device, pinned: bool, fill: int = 0) -> torch.Tensor:
    if pinned:
        t = torch.empty(n, dtype=dtype, pin_memory=True)
        t.fill_(fill - 65536 if (dtype == torch.int16 and fill >= 32768) else fill)
        return t
    if dtype == torch.int16:
        return _u16_empty(n, device, fill)
    return torch.full((n,), float(fill), dtype=dtype, device=device)


class NadamGroup(_Group):
    """Kahan + u16-moment NAdam(W)/Adam state for a list of bf16 weights (one library group).
    With `offload`, residuals and moments live in pinned host memory and move through the
    engine's staging slots around each step."""

    kind = lmopt.OPTIM_KIND_NADAM

    def __init__(self, weights: Sequence[torch.Tensor], residuals: Sequence[torch.Tensor] | None = None,
                 kahan: bool = True, offload: OffloadEngine | None = None, states: str = "u16"):
        super().__init__()
        self.weights = list(weights)
        for w in self.weights:
            assert w.dtype == torch.bfloat16 and w.is_cuda and w.is_contiguous()
        dev = self.weights[0].device
        pinned = offload is not None
        assert states in ("u16", "f24")
        self.kind = lmopt.OPTIM_KIND_NADAM_F24 if states == "f24" else lmopt.OPTIM_KIND_NADAM
        if residuals is None:
            residuals = [_state_buffer(w.numel(), torch.int16, dev, pinned) if kahan else None for w in self.weights]
        elif pinned:
            residuals = [r.cpu().pin_memory() if r is not None else None for r in residuals]
        self.res = list(residuals)
        self.m, self.v = [], []
        for w in self.weights:
            n = w.numel()
            if n <= SMALL:
                self.m.append(_state_buffer(n, torch.float32, dev, pinned))
                self.v.append(_state_buffer(n, torch.float32, dev, pinned))
            elif states == "f24":       # n upper 16-bit words, padding to 16 B, n low bytes, all zero
                nbytes = (2 * n + 15) // 16 * 16 + n
                self.m.append(_state_buffer(nbytes, torch.uint8, dev, pinned))
                self.v.append(_state_buffer(nbytes, torch.uint8, dev, pinned))
            else:
                self.m.append(_state_buffer(n, torch.int16, dev, pinned, 32768))
                self.v.append(_state_buffer(n, torch.int16, dev, pinned, 0))
        descs = [_desc(w, r, m, v, w.shape) for w, r, m, v in zip(self.weights, self.res, self.m, self.v)]
        self.handle = lmopt.optim_group_create(descs, self.kind)
        self.offload = offload
        if offload is not None:
            lmopt.optim_group_attach_offload(self.handle, offload.handle)

    @classmethod
    def from_masters(cls, masters: Sequence[torch.Tensor], stream=None, offload: OffloadEngine | None = None,
                     states: str = "u16"):
        ws, rs = [], []
        for x in masters:
            hi, lo = kahan_split(x.contiguous(), stream=stream)
            ws.append(hi)
            rs.append(lo)
        return cls(ws, rs, offload=offload, states=states)

    @staticmethod
    def _hparams(hp: dict) -> lmopt.NadamHparams:
        return lmopt.NadamHparams(lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"],
                                  weight_decay=hp.get("weight_decay", 0.0), wd_mode=hp.get("wd_mode", 0),
                                  nesterov=hp.get("nesterov", 1), momentum_decay=hp.get("momentum_decay", 0.004),
                                  stochastic_rounding=hp.get("stochastic_rounding", 0), seed=hp.get("seed", 0))

    def step(self, grads: Sequence[torch.Tensor], hp: dict, stream=None):
        lmopt.optim_step_nadam_kahan(self.handle, self._grad_ptrs(grads), self.step_count + 1, self._hparams(hp),
                                     _stream_ptr(stream))
        self.step_count += 1

    def launches(self, hp: dict) -> int:
        """Kernel launches one step enqueues (1 for groups small enough for the one-launch step)."""
        return lmopt.optim_query_launches(self.handle, self._hparams(hp))

    def exchange_buffer(self) -> torch.Tensor:
        """Device buffer of 3 floats per tensor for optim_step_nadam_begin / _end."""
        return torch.zeros(3 * len(self.weights), dtype=torch.float32, device=self.weights[0].device)

    def step_begin(self, grads: Sequence[torch.Tensor], hp: dict, exchange: torch.Tensor | None = None, stream=None):
        """Gradient pre-pass; fills `exchange` with the per-tensor maxima to MAX-reduce across ranks."""
        lmopt.optim_step_nadam_begin(self.handle, self._grad_ptrs(grads), self.step_count + 1, self._hparams(hp),
                                     _stream_ptr(stream), exchange.data_ptr() if exchange is not None else None)

    def step_end(self, exchange: torch.Tensor | None = None, stream=None):
        """Update, after the reduced maxima are written back from `exchange`."""
        lmopt.optim_step_nadam_end(self.handle, exchange.data_ptr() if exchange is not None else None,
                                   _stream_ptr(stream))
        self.step_count += 1

    def masters(self):
        return [kahan_merge(w, r.to(w.device)) for w, r in zip(self.weights, self.res)]

    def scales(self):
        return lmopt.optim_query_scales(self.handle, len(self.weights))


class FactoredGroup(_Group):
    """Adafactor / Prodigy factored-second-moment state (beta1 = 0, no exp_avg)."""

    kind = lmopt.OPTIM_KIND_FACTORED

    def __init__(self, weights: Sequence[torch.Tensor], residuals: Sequence[torch.Tensor] | None = None,
                 kahan: bool = True):
        super().__init__()
        self.weights = list(weights)
        dev = self.weights[0].device
        if residuals is None:
            residuals = [_u16_empty(w.numel(), dev, 0) if kahan else None for w in self.weights]
        self.res = list(residuals)
        self.row, self.col = [], []
        for w in self.weights:
            shape = tuple(w.shape)
            if len(shape) >= 2:
                lead = int(torch.tensor(shape[:-2]).prod().item()) if len(shape) > 2 else 1
                self.row.append(torch.zeros(lead * shape[-2], dtype=torch.float32, device=dev))
                self.col.append(torch.zeros(lead * shape[-1], dtype=torch.float32, device=dev))
            else:
                self.row.append(None)
                self.col.append(torch.zeros(w.numel(), dtype=torch.float32, device=dev))
        descs = [_desc(w, r, m, v, w.shape) for w, r, m, v in zip(self.weights, self.res, self.row, self.col)]
        self.handle = lmopt.optim_group_create(descs, self.kind)

    @classmethod
    def from_masters(cls, masters: Sequence[torch.Tensor], stream=None):
        ws, rs = [], []
        for x in masters:
            hi, lo = kahan_split(x.contiguous(), stream=stream)
            ws.append(hi)
            rs.append(lo)
        return cls(ws, rs)

    def step(self, grads: Sequence[torch.Tensor], hp: dict, stream=None):
        h = lmopt.FactoredHparams(lr=hp["lr"], beta2=hp.get("beta2", 0.999), decay_rate=hp.get("decay_rate", -0.8),
                                  eps1=hp.get("eps1", 1e-30), eps2=hp.get("eps2", 1e-30), d=hp.get("d", 1.0),
                                  clip_threshold=hp.get("clip_threshold", 1.0),
                                  weight_decay=hp.get("weight_decay", 0.0), mode=hp.get("mode", 0))
        lmopt.optim_step_factored(self.handle, self._grad_ptrs(grads), self.step_count + 1, h, _stream_ptr(stream))
        self.step_count += 1

    def masters(self):
        return [kahan_merge(w, r) for w, r in zip(self.weights, self.res)]

    def attach_prodigy(self, ctrl: "ProdigyController", stream=None, p0=None, s=None):
        """Shares d with every other group of `ctrl`: allocates the sampled p0 / s buffers and
        snapshots the current weights into p0, or (p0 and s given, e.g. from a checkpoint)
        takes copies of them as they are; later steps use mode 1 with the controller's d."""
        dev = self.weights[0].device
        restore = p0 is not None
        src_p0, src_s = p0, s
        p0, s = [], []
        for i, w in enumerate(self.weights):
            n = lmopt.optim_prodigy_slice_len(w.numel(), ctrl.slice_p)
            if restore:
                assert src_p0[i].numel() == max(n, 1) and src_s[i].numel() == max(n, 1)
                p0.append(src_p0[i].to(dev, torch.float32).clone())
                s.append(src_s[i].to(dev, torch.float32).clone())
            else:
                p0.append(torch.zeros(max(n, 1), dtype=torch.float32, device=dev))
                s.append(torch.zeros(max(n, 1), dtype=torch.float32, device=dev))
        lmopt.optim_group_attach_prodigy(self.handle, ctrl.handle, [t.data_ptr() for t in p0],
                                         [t.data_ptr() for t in s], 0 if restore else 1, _stream_ptr(stream))
        self.p0, self.s = p0, s     # kept alive while attached
        ctrl.groups.append(self)


class ProdigyController:
    """Prodigy's step-size estimate d shared by the FACTORED groups attached to it: step every
    group (mode 1), then call end_step() once.  close() destroys the attached groups as well (the
    controller cannot be freed while groups are attached)."""

    def __init__(self, d0: float = 1e-6, beta3: float | None = None, beta2: float = 0.999, slice_p: int = 11):
        self.slice_p = slice_p
        self.beta3 = float(beta3) if beta3 is not None else float(beta2) ** 0.5
        self.handle = lmopt.optim_prodigy_create(d0, self.beta3, slice_p)
        self.groups = []

    def end_step(self, stream=None, all_reduce_sum=None):
        """After every attached group stepped.  With data-parallel processes that share d, pass
        all_reduce_sum (a callable SUM-reducing a float64 device tensor in place, e.g.
        torch.distributed.all_reduce): this process's two sums are reduced across processes
        before d is updated."""
        if all_reduce_sum is None:
            lmopt.optim_prodigy_end_step(self.handle, _stream_ptr(stream))
            return
        dev = self.groups[0].weights[0].device if self.groups else torch.device("cuda")
        buf = torch.empty(2, dtype=torch.float64, device=dev)
        lmopt.optim_prodigy_reduce(self.handle, buf.data_ptr(), _stream_ptr(stream))
        all_reduce_sum(buf)
        lmopt.optim_prodigy_finish(self.handle, buf.data_ptr(), _stream_ptr(stream))

    def get(self):
        return lmopt.optim_prodigy_get(self.handle)

    def set(self, d: float, r: float):
        lmopt.optim_prodigy_set(self.handle, d, r)

    def close(self):
        if self.handle:
            for g in self.groups:
                g.close()
            self.groups = []
            lmopt.optim_prodigy_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def adan_f24_stride(n: int) -> int:
    """Bytes between the m, v and n f24 buffers of an ADAN_F24 state: f24 bytes rounded up to 16."""
    return ((2 * n + 15) // 16 * 16 + n + 15) // 16 * 16


class AdanGroup(_Group):
    """Adan state (m, v, n and the previous bf16 gradient) for a list of bf16 weights: fp32 planes,
    or with states="f24" three f24 buffers for tensors above 4096 elements.  With `offload`
    (an OffloadEngine) the residuals and states live in pinned host memory."""

    kind = lmopt.OPTIM_KIND_ADAN
    _state_attrs = ("res", "mvn", "gprev")

    def __init__(self, weights: Sequence[torch.Tensor], residuals: Sequence[torch.Tensor] | None = None,
                 kahan: bool = True, states: str = "fp32", offload: OffloadEngine | None = None):
        super().__init__()
        assert states in ("fp32", "f24")
        self.kind = lmopt.OPTIM_KIND_ADAN_F24 if states == "f24" else lmopt.OPTIM_KIND_ADAN
        self.weights = list(weights)
        dev = self.weights[0].device
        pinned = offload is not None
        if residuals is None:
            residuals = [_state_buffer(w.numel(), torch.int16, dev, pinned) if kahan else None for w in self.weights]
        elif pinned:
            residuals = [r.cpu().pin_memory() if r is not None else None for r in residuals]
        self.res = list(residuals)
        # planes m, v, n, each numel rounded up to a multiple of 4 floats (16-byte aligned planes);
        # f24: three f24 buffers of adan_f24_stride bytes each
        self.mvn = []
        for w in self.weights:
            n = w.numel()
            if states == "f24" and n > SMALL:
                self.mvn.append(_state_buffer(3 * adan_f24_stride(n), torch.uint8, dev, pinned))
            else:
                self.mvn.append(_state_buffer(3 * ((n + 3) // 4 * 4), torch.float32, dev, pinned))
        self.gprev = [_state_buffer(w.numel(), torch.int16, dev, pinned) for w in self.weights]
        descs = [_desc(w, r, m, v, w.shape) for w, r, m, v in zip(self.weights, self.res, self.mvn, self.gprev)]
        self.handle = lmopt.optim_group_create(descs, self.kind)
        self.offload = offload
        if offload is not None:
            lmopt.optim_group_attach_offload(self.handle, offload.handle)

    @classmethod
    def from_masters(cls, masters: Sequence[torch.Tensor], stream=None, states: str = "fp32",
                     offload: OffloadEngine | None = None):
        ws, rs = [], []
        for x in masters:
            hi, lo = kahan_split(x.contiguous(), stream=stream)
            ws.append(hi)
            rs.append(lo)
        return cls(ws, rs, states=states, offload=offload)

    def step(self, grads: Sequence[torch.Tensor], hp: dict, stream=None):
        h = lmopt.AdanHparams(lr=hp["lr"], beta1=hp.get("beta1", 0.02), beta2=hp.get("beta2", 0.08),
                              beta3=hp.get("beta3", 0.01), eps=hp.get("eps", 1e-8),
                              weight_decay=hp.get("weight_decay", 0.0),
                              stochastic_rounding=hp.get("stochastic_rounding", 0), seed=hp.get("seed", 0))
        lmopt.optim_step_adan(self.handle, self._grad_ptrs(grads), self.step_count + 1, h, _stream_ptr(stream))
        self.step_count += 1

    def masters(self):
        return [kahan_merge(w, r.to(w.device)) for w, r in zip(self.weights, self.res)]
