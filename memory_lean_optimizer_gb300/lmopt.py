"""Thin ctypes binding of liblmopt.so (include/lmopt.h): argument marshalling only.

Every function here has the name of its C entry point and takes plain integers for device
pointers (``tensor.data_ptr()``) and streams (``torch.cuda.Stream.cuda_stream``); all work runs in
the library's CUDA kernels.  The library must have been built (``memory_lean_optimizer_gb300.build``):
there is no fallback, and a missing library raises at first use.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "liblmopt.so")

OPTIM_OK = 0
OPTIM_EINVAL = -1
OPTIM_ECUDA = -2
OPTIM_ENOMEM = -3
OPTIM_EALIGN = -4
OPTIM_ETIMEOUT = -5
OPTIM_ENONFINITE = -6
OPTIM_ESTATE = -7
OPTIM_KIND_NADAM = 0
OPTIM_KIND_FACTORED = 1
OPTIM_KIND_NADAM_F24 = 2
OPTIM_KIND_ADAN = 3
OPTIM_KIND_ADAN_F24 = 4
SMALL_NUMEL = 4096

ERROR_NAMES = {OPTIM_EINVAL: "EINVAL", OPTIM_ECUDA: "ECUDA", OPTIM_ENOMEM: "ENOMEM", OPTIM_EALIGN: "EALIGN",
               OPTIM_ETIMEOUT: "ETIMEOUT", OPTIM_ENONFINITE: "ENONFINITE", OPTIM_ESTATE: "ESTATE"}

EXPORTED = (
    "optim_group_create", "optim_group_destroy", "optim_step_nadam_kahan", "optim_step_factored",
    "state_pack_u16", "state_unpack_u16", "optim_kahan_split", "optim_kahan_merge",
    "optim_query_scales", "optim_set_scales", "optim_group_get_step", "optim_group_set_step",
    "optim_query_nonfinite", "optim_group_set_profile_event", "optim_last_error",
    "optim_step_factored_noalloc", "optim_step_adan",
    "optim_offload_create", "optim_offload_destroy", "optim_group_attach_offload",
    "optim_offload_prefetch", "optim_offload_sync", "optim_offload_writeback", "optim_group_attach_host",
    "optim_offload_layout", "optim_step_nadam_begin", "optim_step_nadam_end", "optim_query_launches",
    "optim_prodigy_create", "optim_prodigy_destroy", "optim_prodigy_slice_len", "optim_group_attach_prodigy",
    "optim_prodigy_end_step", "optim_prodigy_get", "optim_prodigy_set", "optim_prodigy_reduce",
    "optim_prodigy_finish",
)


class LmoptError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class TensorDesc(ctypes.Structure):
    _fields_ = [("w_bf16", ctypes.c_void_p), ("res_u16", ctypes.c_void_p), ("m", ctypes.c_void_p),
                ("v", ctypes.c_void_p), ("numel", ctypes.c_int64), ("ndim", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("shape", ctypes.c_int64 * 4)]


class NadamHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("wd_mode", ctypes.c_int32),
                ("nesterov", ctypes.c_int32), ("momentum_decay", ctypes.c_float),
                ("stochastic_rounding", ctypes.c_int32), ("seed", ctypes.c_uint64)]


class AdanHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("beta3", ctypes.c_float), ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("stochastic_rounding", ctypes.c_int32), ("reserved", ctypes.c_int32), ("seed", ctypes.c_uint64)]


class FactoredHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta2", ctypes.c_float), ("decay_rate", ctypes.c_float),
                ("eps1", ctypes.c_float), ("eps2", ctypes.c_float), ("d", ctypes.c_float),
                ("clip_threshold", ctypes.c_float), ("weight_decay", ctypes.c_float), ("mode", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Loads liblmopt.so (once) and declares its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m memory_lean_optimizer_gb300.build` "
                               "(the engine has no CPU fallback)")
        lib = ctypes.CDLL(path)
        P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        sig = {
            "optim_group_create": [ctypes.POINTER(TensorDesc), I32, I32, ctypes.POINTER(P)],
            "optim_group_destroy": [P],
            "optim_step_nadam_kahan": [P, P, I64, ctypes.POINTER(NadamHparams), P],
            "optim_step_nadam_begin": [P, P, I64, ctypes.POINTER(NadamHparams), P, P],
            "optim_step_nadam_end": [P, P, P],
            "optim_step_factored": [P, P, I64, ctypes.POINTER(FactoredHparams), P],
            "optim_step_adan": [P, P, I64, ctypes.POINTER(AdanHparams), P],
            "optim_step_factored_noalloc": [ctypes.POINTER(TensorDesc), P, I64, ctypes.POINTER(FactoredHparams), P],
            "state_pack_u16": [P, P, P, I64, I32, P],
            "state_unpack_u16": [P, P, P, I64, I32, P],
            "optim_kahan_split": [P, P, P, I64, P],
            "optim_kahan_merge": [P, P, P, I64, P],
            "optim_query_scales": [P, P],
            "optim_set_scales": [P, P],
            "optim_group_get_step": [P, ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_double)],
            "optim_group_set_step": [P, I64, ctypes.c_double],
            "optim_query_nonfinite": [P, ctypes.POINTER(ctypes.c_uint64)],
            "optim_query_launches": [P, P, ctypes.POINTER(I32)],
            "optim_group_set_profile_event": [P, P],
            "optim_offload_create": [ctypes.c_size_t, I32, ctypes.POINTER(P)],
            "optim_offload_destroy": [P],
            "optim_group_attach_offload": [P, P],
            "optim_offload_prefetch": [P, P],
            "optim_offload_writeback": [P, P],
            "optim_group_attach_host": [P, P, ctypes.c_size_t],
            "optim_offload_layout": [P, ctypes.POINTER(I64), ctypes.POINTER(I64)],
            "optim_offload_sync": [P, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)],
            "optim_prodigy_create": [ctypes.c_double, F, I32, ctypes.POINTER(P)],
            "optim_prodigy_destroy": [P],
            "optim_group_attach_prodigy": [P, P, P, P, I32, P],
            "optim_prodigy_end_step": [P, P],
            "optim_prodigy_reduce": [P, P, P],
            "optim_prodigy_finish": [P, P, P],
            "optim_prodigy_get": [P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)],
            "optim_prodigy_set": [P, ctypes.c_double, ctypes.c_double],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.optim_prodigy_slice_len.argtypes = [I64, I32]
        lib.optim_prodigy_slice_len.restype = I64
        lib.optim_last_error.argtypes = []
        lib.optim_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def last_error() -> str:
    return load().optim_last_error().decode()


def check(rc: int) -> int:
    if rc != OPTIM_OK:
        raise LmoptError(rc, last_error())
    return rc


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = p
    return arr


# ------------------------------------------------------------------ raw entry points (same names)
def optim_group_create(descs, kind: int) -> int:
    """descs: sequence of TensorDesc; returns the opaque handle as an int."""
    arr = (TensorDesc * len(descs))(*descs)
    out = ctypes.c_void_p()
    check(load().optim_group_create(arr, len(descs), kind, ctypes.byref(out)))
    return out.value


def optim_group_destroy(handle: int) -> None:
    check(load().optim_group_destroy(handle))


def optim_step_nadam_kahan(handle: int, grad_ptrs, step: int, hp: NadamHparams, stream: int = 0) -> None:
    check(load().optim_step_nadam_kahan(handle, _ptr_array(grad_ptrs), step, ctypes.byref(hp), stream))


def optim_step_nadam_begin(handle: int, grad_ptrs, step: int, hp: NadamHparams, stream: int = 0,
                           exchange: int | None = None) -> None:
    """Pre-pass of a step; with `exchange` (device pointer, 3 floats per tensor) the per-tensor
    maxima to be MAX-reduced across ranks are copied there."""
    check(load().optim_step_nadam_begin(handle, _ptr_array(grad_ptrs), step, ctypes.byref(hp), stream, exchange))


def optim_step_nadam_end(handle: int, exchange: int | None = None, stream: int = 0) -> None:
    """Update of the step begun by optim_step_nadam_begin, after writing back the reduced maxima."""
    check(load().optim_step_nadam_end(handle, exchange, stream))


def optim_step_factored(handle: int, grad_ptrs, step: int, hp: FactoredHparams, stream: int = 0) -> None:
    check(load().optim_step_factored(handle, _ptr_array(grad_ptrs), step, ctypes.byref(hp), stream))


def optim_step_factored_noalloc(desc: TensorDesc, grad_ptr: int, step: int, hp: FactoredHparams,
                                stream: int = 0) -> None:
    """Single-tensor factored step using the library's fixed device scratch (no allocation)."""
    check(load().optim_step_factored_noalloc(ctypes.byref(desc), grad_ptr, step, ctypes.byref(hp), stream))


def optim_step_adan(handle: int, grad_ptrs, step: int, hp: AdanHparams, stream: int = 0) -> None:
    check(load().optim_step_adan(handle, _ptr_array(grad_ptrs), step, ctypes.byref(hp), stream))


def state_pack_u16(src: int, codes: int, scale: int, n: int, is_signed: bool, stream: int = 0) -> None:
    check(load().state_pack_u16(src, codes, scale, n, int(is_signed), stream))


def state_unpack_u16(codes: int, scale: int, dst: int, n: int, is_signed: bool, stream: int = 0) -> None:
    check(load().state_unpack_u16(codes, scale, dst, n, int(is_signed), stream))


def optim_kahan_split(src: int, hi: int, lo: int, n: int, stream: int = 0) -> None:
    check(load().optim_kahan_split(src, hi, lo, n, stream))


def optim_kahan_merge(hi: int, lo: int, dst: int, n: int, stream: int = 0) -> None:
    check(load().optim_kahan_merge(hi, lo, dst, n, stream))


def optim_query_scales(handle: int, n: int):
    """Returns a list of (S_m, S_v, A_m, A_v) per tensor after the last completed step."""
    buf = (ctypes.c_float * (4 * n))()
    check(load().optim_query_scales(handle, buf))
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]


def optim_set_scales(handle: int, records) -> None:
    flat = [float(x) for r in records for x in r]
    buf = (ctypes.c_float * len(flat))(*flat)
    check(load().optim_set_scales(handle, buf))


def optim_group_get_step(handle: int):
    step, mp = ctypes.c_int64(), ctypes.c_double()
    check(load().optim_group_get_step(handle, ctypes.byref(step), ctypes.byref(mp)))
    return step.value, mp.value


def optim_group_set_step(handle: int, step: int, mu_product: float) -> None:
    check(load().optim_group_set_step(handle, step, mu_product))


def optim_group_set_profile_event(handle: int, event: int | None) -> None:
    """event: a cudaEvent_t as int (torch.cuda.Event.cuda_event), or None to turn the hook off."""
    check(load().optim_group_set_profile_event(handle, event))


def optim_query_nonfinite(handle: int) -> int:
    c = ctypes.c_uint64()
    check(load().optim_query_nonfinite(handle, ctypes.byref(c)))
    return c.value


def optim_query_launches(handle: int, hp: NadamHparams | None = None) -> int:
    """Kernel launches one step of the group enqueues (hp: the NAdam hyper-parameters, for NADAM groups)."""
    n = ctypes.c_int32()
    check(load().optim_query_launches(handle, ctypes.byref(hp) if hp is not None else None, ctypes.byref(n)))
    return n.value


def optim_offload_create(slot_bytes: int, n_slots: int) -> int:
    out = ctypes.c_void_p()
    check(load().optim_offload_create(slot_bytes, n_slots, ctypes.byref(out)))
    return out.value


def optim_offload_destroy(engine: int) -> None:
    check(load().optim_offload_destroy(engine))


def optim_group_attach_offload(handle: int, engine: int) -> None:
    check(load().optim_group_attach_offload(handle, engine))


def optim_offload_prefetch(handle: int, copy_stream: int = 0) -> None:
    """Copy-in of an offloaded group's states on `copy_stream` (0: the library's own H2D stream)."""
    check(load().optim_offload_prefetch(handle, copy_stream))


def optim_offload_writeback(handle: int, copy_stream: int = 0) -> None:
    """Copy-out after the group's last step on `copy_stream` (0: the library's own D2H stream)."""
    check(load().optim_offload_writeback(handle, copy_stream))


def optim_offload_layout(handle: int, n_tensors: int):
    """(total bytes of the group's host image, [(res, m, v) byte offsets per tensor, -1 if absent])."""
    offs = (ctypes.c_int64 * max(1, 3 * n_tensors))()
    total = ctypes.c_int64()
    check(load().optim_offload_layout(handle, offs, ctypes.byref(total)))
    return total.value, [tuple(offs[3 * i:3 * i + 3]) for i in range(n_tensors)]


def optim_group_attach_host(handle: int, image_ptr: int, nbytes: int) -> None:
    check(load().optim_group_attach_host(handle, image_ptr, nbytes))


def optim_offload_sync(engine: int | None):
    """Returns (bytes copied host->device, bytes copied device->host) so far; engine None: the
    library's own staging ring of the current device."""
    a, b = ctypes.c_uint64(), ctypes.c_uint64()
    check(load().optim_offload_sync(engine, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def optim_prodigy_create(d0: float, beta3: float, slice_p: int) -> int:
    out = ctypes.c_void_p()
    check(load().optim_prodigy_create(d0, beta3, slice_p, ctypes.byref(out)))
    return out.value


def optim_prodigy_destroy(pd: int) -> None:
    check(load().optim_prodigy_destroy(pd))


def optim_prodigy_slice_len(numel: int, slice_p: int) -> int:
    return int(load().optim_prodigy_slice_len(numel, slice_p))


def optim_group_attach_prodigy(handle: int, pd: int, p0_ptrs, s_ptrs, snapshot: int = 1, stream: int = 0) -> None:
    n = len(p0_ptrs)
    a = (ctypes.c_void_p * max(n, 1))(*p0_ptrs)
    b = (ctypes.c_void_p * max(n, 1))(*s_ptrs)
    check(load().optim_group_attach_prodigy(handle, pd, a, b, int(snapshot), stream))


def optim_prodigy_end_step(pd: int, stream: int = 0) -> None:
    check(load().optim_prodigy_end_step(pd, stream))


def optim_prodigy_reduce(pd: int, partial_ptr: int, stream: int = 0) -> None:
    check(load().optim_prodigy_reduce(pd, partial_ptr, stream))


def optim_prodigy_finish(pd: int, total_ptr: int, stream: int = 0) -> None:
    check(load().optim_prodigy_finish(pd, total_ptr, stream))


def optim_prodigy_get(pd: int):
    """(d, r) of the controller (synchronises the device)."""
    d, r = ctypes.c_double(), ctypes.c_double()
    check(load().optim_prodigy_get(pd, ctypes.byref(d), ctypes.byref(r)))
    return d.value, r.value


def optim_prodigy_set(pd: int, d: float, r: float) -> None:
    check(load().optim_prodigy_set(pd, d, r))
