"""CPU oracle of the fused optimizer step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It wraps ``oracle.c`` (plain single-threaded C, compiled with gcc and
``-ffp-contract=off``) through ctypes and numpy; it shares no code with the CUDA library.

Parity status of each function (pins live in ``tests/test_oracle_*.py``):
  kahan_split / kahan_merge      pinned: exhaustive 2^32 round trip, IEEE bit-pattern fixtures
  round_bf16                     pinned: torch's round-to-nearest-even bf16 cast
  encode/decode (u16 codec)      pinned: exhaustive 65536-code round trip, half-step bound,
                                 monotonicity, hand-derived fixtures (tie to even)
  nadam_scalars / nadam_step     pinned: Adam step-1 = -lr sign(g), NAdam step-1 closed form,
                                 torch.optim.Adam/AdamW/NAdam trajectories, zero grad, decay-only
  scale record (S_m, S_v, A_m, A_v)  pinned: closed forms at t = 1 (S = (1-b) G, (1-b2) G^2) and
                                 the recurrence at t = 2 on hand-chosen maxima, both store paths
  nadam_step_slice               pinned: slices stepped with the whole tensor's maxima equal the
                                 unsplit step (gloo tests)
  nadam_step_tensor_f24          pinned: replay of the fp32-moment step truncated to 24 bits,
                                 2^-15 storage bound, hand-computed plane layout
  philox4x32_10 / sr_bits / stochastic_round / nadam_step_tensor_sr
                                 pinned: the generator's published known-answer vectors, lane
                                 uniformity, rounding probability equal to the distance, SR step
                                 = RNE-free rounding of the no-residual step
  adan_step_tensor               pinned: constant-gradient and two-gradient closed forms, decay only
  factored_step                  pinned: torch.optim.Adafactor special case, rank-1 g^2 gives
                                 u = sign(g), 1-D step-1 sign, clipped RMS == clip, zero grad
  prodigy_* (d estimate)         pinned: closed-form numerator at t = 1, constant-gradient scalar
                                 recurrence, slicing independence, monotone d
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_LIB_MT_PATH = os.path.join(_OUT_DIR, "liboracle_mt.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall",
           "-Wno-unknown-pragmas"]

_lock = threading.Lock()
_lib = None
_lib_mt = None

SMALL_NUMEL = 4096


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, single-threaded: the parity
    reference) and, from the same source with OpenMP, liboracle_mt.so (its threaded timing driver;
    without OpenMP in the compiler it is built single-threaded); returns the first path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    for path, extra in ((_LIB_PATH, []), (_LIB_MT_PATH, ["-fopenmp"])):
        if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
            tmp = path + f".tmp{os.getpid()}"
            try:
                subprocess.check_call(["gcc", *_CFLAGS, *extra, "-o", tmp, _SRC, "-lm"])
            except subprocess.CalledProcessError:
                if not extra:
                    raise
                subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, path)
    return _LIB_PATH


class NadamScalars(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in
                ("lr", "b1", "omb1", "b2", "omb2", "eps", "lr_wd", "c_m", "c_g", "k2")] + \
               [("decoupled_wd", ctypes.c_int32)]


class Scale(ctypes.Structure):
    _fields_ = [("s_m", ctypes.c_float), ("s_v", ctypes.c_float),
                ("a_m", ctypes.c_float), ("a_v", ctypes.c_float)]


class CodecConsts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in ("qm", "rm", "qv", "rv")]


class AdanScalars(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in ("lr", "b1", "omb1", "b2", "omb2", "b3", "omb3", "eps", "inv_decay")]


class FactoredScalars(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in
                ("b2t", "alpha", "eps1", "eps2", "clip", "lr_eff", "nwdlr")] + \
               [("mode", ctypes.c_int32), ("unum", ctypes.c_float)]


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        F = ctypes.c_float
        I32 = ctypes.c_int32
        sig = {
            "orc_kahan_split": (None, [P, P, P, I64]),
            "orc_kahan_merge": (None, [P, P, P, I64]),
            "orc_round_bf16": (None, [P, P, I64]),
            "orc_codec_consts": (None, [F, F, ctypes.POINTER(CodecConsts)]),
            "orc_encode_m": (ctypes.c_uint16, [F, F]),
            "orc_decode_m": (F, [ctypes.c_uint16, F]),
            "orc_encode_v": (ctypes.c_uint16, [F, F]),
            "orc_decode_v": (F, [ctypes.c_uint16, F]),
            "orc_state_pack": (None, [P, P, P, I64, I32]),
            "orc_state_unpack": (None, [P, F, P, I64, I32]),
            "orc_nadam_scalars": (None, [I64, F, F, F, F, F, I32, I32, F,
                                         ctypes.POINTER(ctypes.c_double), ctypes.POINTER(NadamScalars)]),
            "orc_grad_absmax": (F, [P, I64]),
            "orc_nadam_step_tensor": (None, [P, P, P, P, P, I64, ctypes.POINTER(Scale),
                                             ctypes.POINTER(NadamScalars)]),
            "orc_nadam_step_slice": (None, [P, P, P, P, P, I64, I32, F, ctypes.POINTER(Scale),
                                            ctypes.POINTER(NadamScalars)]),
            "orc_nadam_step_fp32": (None, [P, P, P, P, I64, ctypes.POINTER(NadamScalars)]),
            "orc_nadam_step_tensor_f24": (None, [P, P, P, P, P, I64, ctypes.POINTER(NadamScalars), I32,
                                                 ctypes.c_uint64, ctypes.c_uint32, I64]),
            "orc_philox4x32_10": (None, [P, P, P]),
            "orc_adan_scalars": (None, [F, F, F, F, F, F, ctypes.POINTER(AdanScalars)]),
            "orc_adan_step_tensor": (None, [P, P, P, P, P, I64, I64, ctypes.POINTER(AdanScalars), I32,
                                            ctypes.c_uint64, ctypes.c_uint32]),
            "orc_adan_step_tensor_f24": (None, [P, P, P, P, P, I64, I64, ctypes.POINTER(AdanScalars), I32,
                                                ctypes.c_uint64, ctypes.c_uint32]),
            "orc_adan_f24_stride": (I64, [I64]),
            "orc_sr_bits": (ctypes.c_uint32, [ctypes.c_uint64, ctypes.c_uint32, I64, I64]),
            "orc_stochastic_round": (None, [P, P, I64, ctypes.c_uint64, ctypes.c_uint32, I64]),
            "orc_nadam_step_tensor_sr": (None, [P, P, P, P, I64, ctypes.POINTER(Scale), ctypes.POINTER(NadamScalars),
                                                ctypes.c_uint64, ctypes.c_uint32, I64]),
            "orc_factored_scalars": (None, [I64, F, F, F, F, F, F, F, F, I32,
                                            ctypes.POINTER(FactoredScalars)]),
            "orc_factored_step_tensor": (F, [P, P, P, I64, I64, I64, P, P,
                                             ctypes.POINTER(FactoredScalars)]),
            "orc_factored_step_vector": (F, [P, P, P, I64, P, ctypes.POINTER(FactoredScalars)]),
            "orc_prodigy_slice_len": (I64, [I64, I32]),
            "orc_prodigy_snapshot": (None, [P, P, I64, I32, P, P]),
            "orc_prodigy_tensor_stats": (None, [P, P, P, I64, I32, P, P, F, F, ctypes.POINTER(ctypes.c_double),
                                                ctypes.POINTER(ctypes.c_double)]),
            "orc_prodigy_end_step": (None, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                            ctypes.c_double, ctypes.c_double, ctypes.c_double]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _load_mt():
    global _lib_mt
    with _lock:
        if _lib_mt is None:
            build()
            lib = ctypes.CDLL(_LIB_MT_PATH)
            lib.orc_threads.argtypes = []
            lib.orc_threads.restype = ctypes.c_int32
            lib.orc_nadam_group_step_mt.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                                    ctypes.POINTER(Scale), ctypes.POINTER(NadamScalars)]
            lib.orc_nadam_group_step_mt.restype = None
            _lib_mt = lib
        return _lib_mt


def threads() -> int:
    """Threads the threaded timing driver uses (OpenMP's default: every host core)."""
    return int(_load_mt().orc_threads())


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags.c_contiguous, "oracle buffers must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16
    return a


# ---------------------------------------------------------------- Kahan split / merge, bf16
def kahan_split(x: np.ndarray, hi: np.ndarray | None = None, lo: np.ndarray | None = None):
    """(hi, lo) halves of each fp32 pattern; hi / lo may be given (contiguous uint16, x's size)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    hi = np.empty(x.shape, np.uint16) if hi is None else hi
    lo = np.empty(x.shape, np.uint16) if lo is None else lo
    assert hi.dtype == lo.dtype == np.uint16 and hi.size == lo.size == x.size and hi.flags.c_contiguous and lo.flags.c_contiguous
    _load().orc_kahan_split(_p(x), _p(hi), _p(lo), x.size)
    return hi, lo


def kahan_merge(hi: np.ndarray, lo: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
    hi, lo = _u16(hi), _u16(lo)
    out = np.empty(hi.shape, np.float32) if out is None else out
    assert out.dtype == np.float32 and out.size == hi.size and out.flags.c_contiguous
    _load().orc_kahan_merge(_p(hi), _p(lo), _p(out), hi.size)
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().orc_round_bf16(_p(x), _p(out), x.size)
    return out


# ---------------------------------------------------------------- u16 codec
def codec_consts(s_m: float, s_v: float) -> CodecConsts:
    """Per-tensor codec constants (qm, rm, qv, rv) from the scales S_m, S_v."""
    c = CodecConsts()
    _load().orc_codec_consts(s_m, s_v, ctypes.byref(c))
    return c


def encode_m(m: float, rm: float) -> int:
    return _load().orc_encode_m(m, rm)


def decode_m(c: int, qm: float) -> float:
    return _load().orc_decode_m(c, qm)


def encode_v(sv: float, rv: float) -> int:
    """sv = sqrt(v)."""
    return _load().orc_encode_v(sv, rv)


def decode_v(c: int, qv: float) -> float:
    return _load().orc_decode_v(c, qv)


def state_pack(x: np.ndarray, is_signed: bool):
    """fp32 moments -> (u16 codes, scale); scale = max |x| (signed) or max x."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.empty(x.shape, np.uint16)
    scale = np.zeros(1, np.float32)
    _load().orc_state_pack(_p(x), _p(codes), _p(scale), x.size, int(is_signed))
    return codes, float(scale[0])


def state_unpack(codes: np.ndarray, scale: float, is_signed: bool) -> np.ndarray:
    codes = _u16(codes)
    out = np.empty(codes.shape, np.float32)
    _load().orc_state_unpack(_p(codes), scale, _p(out), codes.size, int(is_signed))
    return out


# ---------------------------------------------------------------- NAdam / Adam
class NadamState:
    """Oracle state of one group: per-tensor scale records plus the NAdam mu product."""

    def __init__(self, n_tensors: int):
        self.scales = (Scale * n_tensors)()
        self.mu_product = ctypes.c_double(1.0)

    def scale(self, i):
        s = self.scales[i]
        return s.s_m, s.s_v, s.a_m, s.a_v


def nadam_scalars(t, lr, beta1, beta2, eps, wd, decoupled_wd, nesterov, psi, mu_product):
    """Returns (NadamScalars, new mu_product)."""
    k = NadamScalars()
    mp = ctypes.c_double(mu_product)
    _load().orc_nadam_scalars(int(t), lr, beta1, beta2, eps, wd, int(decoupled_wd), int(nesterov),
                              psi, ctypes.byref(mp), ctypes.byref(k))
    return k, mp.value


def grad_absmax(g: np.ndarray) -> float:
    g = _u16(g)
    return _load().orc_grad_absmax(_p(g), g.size)


def nadam_step_tensor(hi, lo, m, v, g, scale: Scale, k: NadamScalars):
    """In place on numpy buffers: hi/lo uint16 (lo may be None), m/v uint16 codes or float32."""
    n = hi.size
    _load().orc_nadam_step_tensor(_p(hi), _p(lo), _p(m), _p(v), _p(_u16(g)), n,
                                  ctypes.byref(scale), ctypes.byref(k))


def nadam_step_tensor_f24(hi, lo, m, v, g, k: NadamScalars, sr=False, seed=0, tensor=0, step=0):
    """f24 moments: m, v are uint8 buffers of f24_nbytes(n) bytes (n uint16 upper words, zero
    padding to byte f24_lo_offset(n), then n low bytes), or float32 arrays when n <= 4096.  sr (lo None): stochastic rounding of the weight."""
    _load().orc_nadam_step_tensor_f24(_p(hi), _p(lo), _p(m), _p(v), _p(_u16(g)), hi.size, ctypes.byref(k),
                                      int(sr), seed, tensor, step)


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, np.uint32)
    k = np.ascontiguousarray(key, np.uint32)
    out = np.zeros(4, np.uint32)
    _load().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_bits(seed, tensor, step, i) -> int:
    return _load().orc_sr_bits(seed, tensor, step, i)


def stochastic_round(x: np.ndarray, seed: int, tensor: int, step: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().orc_stochastic_round(_p(x), _p(out), x.size, seed, tensor, step)
    return out


def nadam_step_tensor_sr(hi, m, v, g, scale: Scale, k: NadamScalars, seed: int, tensor: int, step: int):
    _load().orc_nadam_step_tensor_sr(_p(hi), _p(m), _p(v), _p(_u16(g)), hi.size, ctypes.byref(scale),
                                     ctypes.byref(k), seed, tensor, step)


def adan_scalars(lr, b1, b2, b3, eps, wd) -> AdanScalars:
    k = AdanScalars()
    _load().orc_adan_scalars(lr, b1, b2, b3, eps, wd, ctypes.byref(k))
    return k


def adan_plane(n: int) -> int:
    """Stride of the m, v, n planes of an Adan state buffer: n rounded up to a multiple of 4."""
    return (n + 3) // 4 * 4


def adan_step_tensor(hi, lo, mnv, gprev, g, step, k: AdanScalars, sr=False, seed=0, tensor=0):
    """In place: hi/lo uint16 (lo may be None), mnv float32 [3 adan_plane(n)] (m, v, n planes),
    gprev uint16."""
    assert mnv.size == 3 * adan_plane(hi.size)
    _load().orc_adan_step_tensor(_p(hi), _p(lo), _p(mnv), _p(gprev), _p(_u16(g)), hi.size, int(step),
                                 ctypes.byref(k), int(sr), seed, tensor)


def adan_f24_stride(n: int) -> int:
    """Bytes between the m, v and n f24 buffers of an Adan f24 state (f24 bytes of n, rounded up
    to 16)."""
    return int(_load().orc_adan_f24_stride(n))


def adan_f24_nbytes(n: int) -> int:
    """Bytes of an Adan f24 state buffer: three f24 buffers above 4096 elements, else the fp32
    planes of adan_step_tensor."""
    return 3 * adan_f24_stride(n) if n > SMALL_NUMEL else 12 * adan_plane(n)


def adan_step_tensor_f24(hi, lo, buf, gprev, g, step, k: AdanScalars, sr=False, seed=0, tensor=0):
    """In place, as adan_step_tensor, with m, v, n stored as f24 in `buf` (uint8,
    adan_f24_nbytes(n) bytes; fp32 planes for 4096 or fewer elements)."""
    assert buf.dtype == np.uint8 and buf.size == adan_f24_nbytes(hi.size)
    _load().orc_adan_step_tensor_f24(_p(hi), _p(lo), _p(buf), _p(gprev), _p(_u16(g)), hi.size, int(step),
                                     ctypes.byref(k), int(sr), seed, tensor)


def f24_lo_offset(n: int) -> int:
    """Byte offset of the bits-8..15 plane in an f24 buffer: 2n rounded up to 16."""
    return (2 * n + 15) // 16 * 16


def f24_nbytes(n: int) -> int:
    return f24_lo_offset(n) + n


def f24_split(x: np.ndarray) -> np.ndarray:
    """fp32 values -> f24 buffer (upper 16 bits plane, zero padding, then bits 8..15 plane)."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).reshape(-1)
    n = b.size
    out = np.zeros(f24_nbytes(n), np.uint8)
    out[:2 * n].view(np.uint16)[:] = (b >> 16).astype(np.uint16)
    out[f24_lo_offset(n):] = ((b >> 8) & 0xFF).astype(np.uint8)
    return out


def f24_merge(buf: np.ndarray, n: int) -> np.ndarray:
    assert buf.size == f24_nbytes(n)
    hi = buf[:2 * n].view(np.uint16).astype(np.uint32)
    lo = buf[f24_lo_offset(n):].astype(np.uint32)
    return ((hi << 16) | (lo << 8)).view(np.float32)


def nadam_step_fp32(w, m, v, g, k: NadamScalars):
    _load().orc_nadam_step_fp32(_p(w), _p(m), _p(v), _p(_u16(g)), w.size, ctypes.byref(k))


def nadam_step_slice(hi, lo, m, v, g, small: bool, G: float, scale: Scale, k: NadamScalars):
    """One slice of a tensor split across ranks: G and the scale record's A_m, A_v are the maxima
    over all slices (in place, as nadam_step_tensor)."""
    n = hi.size
    _load().orc_nadam_step_slice(_p(hi), _p(lo), _p(m), _p(v), _p(_u16(g)), n, int(small), float(G),
                                 ctypes.byref(scale), ctypes.byref(k))


def nadam_group_step(tensors, grads, state: NadamState, t, hp):
    """One step of a group.  tensors: list of dicts with hi, lo, m, v numpy arrays (in place);
    grads: list of uint16 arrays; hp: dict lr, beta1, beta2, eps, weight_decay, wd_mode,
    nesterov, momentum_decay."""
    k, state.mu_product.value = nadam_scalars(
        t, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"],
        hp["wd_mode"] == 1, hp["nesterov"], hp["momentum_decay"], state.mu_product.value)
    for i, (tt, g) in enumerate(zip(tensors, grads)):
        nadam_step_tensor(tt["hi"], tt.get("lo"), tt["m"], tt["v"], g, state.scales[i], k)
    return k


def nadam_group_step_mt(tensors, grads, state: NadamState, t, hp):
    """nadam_group_step on all host threads (the threaded timing driver of oracle.c): every
    element is updated by the same single-threaded step function on a slice of its tensor, so the
    results are bit-identical to nadam_group_step."""
    k, state.mu_product.value = nadam_scalars(
        t, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"],
        hp["wd_mode"] == 1, hp["nesterov"], hp["momentum_decay"], state.mu_product.value)
    n = len(tensors)
    ptrs = (ctypes.c_void_p * (5 * max(n, 1)))()
    sizes = (ctypes.c_int64 * max(n, 1))()
    keep = []
    for i, (tt, g) in enumerate(zip(tensors, grads)):
        g = _u16(g)
        keep.append(g)
        for j, a in enumerate((tt["hi"], tt.get("lo"), tt["m"], tt["v"], g)):
            ptrs[5 * i + j] = _p(a)
        sizes[i] = tt["hi"].size
    _load_mt().orc_nadam_group_step_mt(n, ptrs, sizes, state.scales, ctypes.byref(k))
    return k


# ---------------------------------------------------------------- factored
def factored_scalars(t, lr, beta2, decay_rate, eps1, eps2, d, clip, wd, mode):
    k = FactoredScalars()
    _load().orc_factored_scalars(int(t), lr, beta2, decay_rate, eps1, eps2, d, clip, wd, int(mode),
                                 ctypes.byref(k))
    return k


def factored_step_tensor(hi, lo, g, B, R, C, row, col, k: FactoredScalars) -> float:
    return _load().orc_factored_step_tensor(_p(hi), _p(lo), _p(_u16(g)), B, R, C, _p(row), _p(col),
                                            ctypes.byref(k))


def factored_step_vector(hi, lo, g, V, k: FactoredScalars) -> float:
    return _load().orc_factored_step_vector(_p(hi), _p(lo), _p(_u16(g)), hi.size, _p(V),
                                            ctypes.byref(k))


# ---------------------------------------------------------------- Prodigy d (R19)
def prodigy_slice_len(n: int, slice_p: int) -> int:
    return _load().orc_prodigy_slice_len(int(n), int(slice_p))


def prodigy_snapshot(hi, lo, slice_p: int):
    """(p0, s) float32 buffers of the sampled elements of the current master."""
    n = hi.size
    L = prodigy_slice_len(n, slice_p)
    p0 = np.zeros(L, np.float32)
    s = np.zeros(L, np.float32)
    _load().orc_prodigy_snapshot(_p(hi), _p(lo), n, int(slice_p), _p(p0), _p(s))
    return p0, s


def prodigy_tensor_stats(hi, lo, g, slice_p, p0, s, beta3, cs):
    """Updates s in place; returns (sum g (p0 - x), sum |s|) of the tensor (before its step)."""
    dot = ctypes.c_double(0.0)
    l1 = ctypes.c_double(0.0)
    _load().orc_prodigy_tensor_stats(_p(hi), _p(lo), _p(_u16(g)), hi.size, int(slice_p), _p(p0), _p(s),
                                     beta3, cs, ctypes.byref(dot), ctypes.byref(l1))
    return dot.value, l1.value


class ProdigyState:
    """d and the numerator r shared by every group of a model (double)."""

    def __init__(self, d0: float, beta3: float, slice_p: int):
        self.d = ctypes.c_double(d0)
        self.r = ctypes.c_double(0.0)
        self.beta3 = float(np.float32(beta3))   # one fp32 beta3 for s and for r
        self.slice_p = slice_p

    def end_step(self, cdot: float, l1: float):
        _load().orc_prodigy_end_step(ctypes.byref(self.d), ctypes.byref(self.r), float(self.beta3), cdot, l1)

    @property
    def d32(self) -> float:
        return float(np.float32(self.d.value))


def prodigy_step(state: ProdigyState, groups, t: int):
    """One step of every group sharing d: prodigy_partials, then the end of the step."""
    cdot, l1 = prodigy_partials(state, groups, t)
    state.end_step(cdot, l1)


def prodigy_partials(state: ProdigyState, groups, t: int):
    """Steps every group with the current d and returns this caller's sums (sum over groups of
    lr d^2 dot, sum |s|) without ending the step.  groups: list of (tensors, grads, hp) where
    each tensor is a dict(hi, lo, shape, row, col or V, p0, s) as for factored_group_step and hp
    the factored hyper-parameters (mode 1; hp["d"] is ignored).  Statistics are taken before each
    tensor's update."""
    d = state.d32
    cdot, l1 = 0.0, 0.0
    beta3 = state.beta3
    for tensors, grads, hp in groups:
        cr = float(np.float32(hp["lr"])) * d * d
        cs = float(np.float32(cr))
        dot_g = 0.0
        for tt, g in zip(tensors, grads):
            dt, lt = prodigy_tensor_stats(tt["hi"], tt.get("lo"), g, state.slice_p, tt["p0"], tt["s"], beta3, cs)
            dot_g += dt
            l1 += lt
        cdot += cr * dot_g
        factored_group_step(tensors, grads, t, dict(hp, d=d, mode=1, decay_rate=hp.get("decay_rate", -0.8)))
    return cdot, l1


def factored_dims(shape):
    """(factored, B, R, C) for a tensor shape: factored over the last two dims iff ndim >= 2."""
    shape = tuple(int(s) for s in shape)
    if len(shape) < 2:
        return False, 1, 1, int(np.prod(shape)) if shape else 1
    B = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
    return True, B, shape[-2], shape[-1]


def factored_group_step(tensors, grads, t, hp):
    """tensors: list of dicts with hi, lo, shape and state 'row','col' (factored) or 'V'."""
    k = factored_scalars(t, hp["lr"], hp["beta2"], hp["decay_rate"], hp["eps1"], hp["eps2"],
                         hp["d"], hp["clip_threshold"], hp["weight_decay"], hp["mode"])
    dens = []
    for tt, g in zip(tensors, grads):
        fac, B, R, C = factored_dims(tt["shape"])
        if fac:
            dens.append(factored_step_tensor(tt["hi"], tt.get("lo"), g, B, R, C, tt["row"], tt["col"], k))
        else:
            dens.append(factored_step_vector(tt["hi"], tt.get("lo"), g, tt["V"], k))
    return k, dens
