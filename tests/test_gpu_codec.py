"""GPU parity of the stand-alone Kahan split/merge and u16 pack/unpack kernels against the oracle,
called through the C ABI.  Bit-exact for every bit pattern and every code."""
import numpy as np
import pytest
import torch

from helpers import alloc_offset

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from memory_lean_optimizer_gb300 import build, lmopt
    build.build()
    lmopt.load()
    return lmopt


def _patterns(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00001, 0x00000001, 0x3F800000,
                        0x3F808000, 0x3F818000, 0xFFFFFFFF, 0x7F7FFFFF], np.uint32)
    bits[:special.size] = special[: min(n, special.size)]
    return bits


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 65536 + 13, 3_000_001])
@pytest.mark.parametrize("offset", [0, 1])
def test_split_merge_bit_exact(lib, orc, n, offset):
    bits = _patterns(n, n + offset)
    x = bits.view(np.float32)
    hi_ref, lo_ref = orc.kahan_split(x)
    _, src = alloc_offset(n, torch.int32, offset)
    src.copy_(torch.from_numpy(bits.view(np.int32)))
    _, hi = alloc_offset(n, torch.int16, offset)
    _, lo = alloc_offset(n, torch.int16, offset)
    lib.optim_kahan_split(src.data_ptr(), hi.data_ptr(), lo.data_ptr(), n, 0)
    torch.cuda.synchronize()
    assert np.array_equal(hi.cpu().numpy().view(np.uint16), hi_ref)
    assert np.array_equal(lo.cpu().numpy().view(np.uint16), lo_ref)
    _, back = alloc_offset(n, torch.int32, offset)
    lib.optim_kahan_merge(hi.data_ptr(), lo.data_ptr(), back.data_ptr(), n, 0)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy().view(np.uint32), bits)


@pytest.mark.parametrize("signed", [True, False])
@pytest.mark.parametrize("n", [1, 4097, 1_000_003])
def test_pack_unpack_bit_exact(lib, orc, signed, n):
    rng = np.random.default_rng(7 + n)
    g = rng.standard_normal(n) * 1e-3
    x = (0.1 * g if signed else 0.001 * g * g).astype(np.float32)
    x[: min(n, 3)] = 0.0
    codes_ref, s_ref = orc.state_pack(x, signed)
    src = torch.from_numpy(x).cuda()
    codes = torch.empty(n, dtype=torch.int16, device="cuda")
    scale = torch.full((1,), 123.0, device="cuda")
    lib.state_pack_u16(src.data_ptr(), codes.data_ptr(), scale.data_ptr(), n, signed, 0)
    torch.cuda.synchronize()
    assert scale.item() == s_ref
    assert np.array_equal(codes.cpu().numpy().view(np.uint16), codes_ref)
    dst = torch.empty(n, dtype=torch.float32, device="cuda")
    lib.state_unpack_u16(codes.data_ptr(), scale.data_ptr(), dst.data_ptr(), n, signed, 0)
    torch.cuda.synchronize()
    ref = orc.state_unpack(codes_ref, s_ref, signed)
    assert np.array_equal(dst.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_every_code_decodes_like_oracle(lib, orc):
    codes = np.arange(65536, dtype=np.uint16)
    c = torch.from_numpy(codes.view(np.int16)).cuda()
    for s in (1e-12, 3.7e-5, 1.0, 2.0 ** 20):
        scale = torch.tensor([s], dtype=torch.float32, device="cuda")
        for signed in (True, False):
            dst = torch.empty(65536, dtype=torch.float32, device="cuda")
            lib.state_unpack_u16(c.data_ptr(), scale.data_ptr(), dst.data_ptr(), 65536, signed, 0)
            torch.cuda.synchronize()
            ref = orc.state_unpack(codes, float(np.float32(s)), signed)
            assert np.array_equal(dst.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_errors_and_empty(lib):
    from memory_lean_optimizer_gb300.lmopt import LmoptError, OPTIM_EINVAL, OPTIM_EALIGN
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")
    lib.optim_kahan_split(0, 0, 0, 0, 0)          # n == 0 is a no-op
    with pytest.raises(LmoptError) as e:
        lib.optim_kahan_split(0, buf.data_ptr(), buf.data_ptr(), 4, 0)
    assert e.value.code == OPTIM_EINVAL
    with pytest.raises(LmoptError) as e:
        lib.optim_kahan_split(buf.data_ptr() + 2, buf.data_ptr(), buf.data_ptr(), 4, 0)
    assert e.value.code == OPTIM_EALIGN
    with pytest.raises(LmoptError) as e:
        lib.state_pack_u16(buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), -1, True, 0)
    assert e.value.code == OPTIM_EINVAL
