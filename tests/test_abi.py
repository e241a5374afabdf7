"""CPU checks of the boundary: liblmopt.so builds (nvcc cross-compiles for sm_103a), loads, and
exports every function include/lmopt.h declares; the ctypes binding covers the same names.
No compute call is made (no GPU here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "lmopt.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib_path():
    from memory_lean_optimizer_gb300 import build
    return build.build()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("optim_step_nadam_kahan", "optim_step_factored", "state_pack_u16", "state_unpack_u16",
                     "optim_kahan_split", "optim_kahan_merge", "optim_group_create", "optim_group_destroy",
                     "optim_group_attach_host", "optim_offload_prefetch", "optim_offload_writeback",
                     "optim_query_scales", "optim_query_nonfinite"):
        assert required in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in lmopt.h but not exported"


def test_binding_covers_header(lib_path):
    from memory_lean_optimizer_gb300 import lmopt
    assert sorted(lmopt.EXPORTED) == declared_functions()
    lib = lmopt.load()
    assert lib.optim_last_error() is not None


def test_invalid_arguments_fail_without_gpu(lib_path):
    """Argument validation happens before any CUDA call, so it is testable on a CPU host."""
    from memory_lean_optimizer_gb300 import lmopt
    lib = lmopt.load()
    assert lib.optim_kahan_split(None, None, None, -1, None) == lmopt.OPTIM_EINVAL
    assert lib.optim_kahan_merge(None, None, None, 0, None) == lmopt.OPTIM_OK
    assert lib.state_pack_u16(None, None, None, 4, 1, None) == lmopt.OPTIM_EINVAL
    assert lib.state_unpack_u16(None, None, None, 4, 2, None) == lmopt.OPTIM_EINVAL
    out = ctypes.c_void_p()
    assert lib.optim_group_create(None, 0, 0, ctypes.byref(out)) == lmopt.OPTIM_EINVAL
    d = lmopt.TensorDesc(numel=10, ndim=1)
    d.shape[0] = 11
    assert lib.optim_group_create(ctypes.byref(d), 1, 0, ctypes.byref(out)) == lmopt.OPTIM_EINVAL
    assert "shape product" in lmopt.last_error()
    d.shape[0] = 10
    d.w_bf16, d.m, d.v = 0x1001, 0x2000, 0x3000
    assert lib.optim_group_create(ctypes.byref(d), 1, 0, ctypes.byref(out)) == lmopt.OPTIM_EALIGN
    assert lib.optim_group_destroy(None) == lmopt.OPTIM_EINVAL
    # the per-group offload calls check their handles first
    assert lib.optim_group_attach_host(None, None, 0) == lmopt.OPTIM_EINVAL
    assert lib.optim_offload_prefetch(None, None) == lmopt.OPTIM_EINVAL
    assert lib.optim_offload_writeback(None, None) == lmopt.OPTIM_EINVAL
    total = ctypes.c_int64()
    assert lib.optim_offload_layout(None, None, ctypes.byref(total)) == lmopt.OPTIM_EINVAL


def test_workload_sizes():
    from memory_lean_optimizer_gb300 import workloads as W
    flux = W.config("flux19")
    assert sum(W.numel(s) for g in flux["groups"] for s in g) == 3_227_516_928
    sd = W.sdxl_like_shapes()
    assert len(sd) == 1332
    assert sum(W.numel(s) for s in sd) == 2_602_705_920
    assert sum(W.numel(s) for g in W.config("flux35")["groups"] for s in g) == 5_945_425_920
    sizes = W.ragged_sizes(20000, 0)
    assert len(sizes) == 20000 and min(sizes) >= 64 and max(sizes) <= 4_194_304
    assert 0.33 < sum(n <= 4096 for n in sizes) / 20000 < 0.42
