"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
symbol include/fp8bs.h declares, and rejects malformed arguments on the host
before touching CUDA (every call here returns before any CUDA runtime call)."""
import ctypes
import os
import re

import pytest
import torch

import fp8_block_scaled_gb300 as fb
from fp8_block_scaled_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID = 0, 1


def _declared_functions():
    names = []
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return fb.load()


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert set(declared) == set(fb.EXPORTS), declared
    handle = ctypes.CDLL(fb.lib_path())
    for name in declared:
        assert hasattr(handle, name), name


def test_library_is_sm103a_only():
    # the build command targets exactly compute_103a / sm_103a
    from fp8_block_scaled_gb300 import build

    assert build.ARCH_FLAGS == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_host_only_entry_points(lib):
    assert fb.abi_version() == 1
    assert fb.status_string(0) == "ok"
    assert "invalid" in fb.status_string(1)
    assert fb.status_string(12345) == "unknown status"
    fb.clear_cache()


def test_debug_flags_take_the_declared_bits_only(lib):
    for flags in (fb.DEBUG_STALL_MMA, fb.DEBUG_SINGLE_CTA, fb.DEBUG_STALL_MMA | fb.DEBUG_SINGLE_CTA, 0):
        assert lib.fp8bs_set_debug_flags(flags) == OK
    assert lib.fp8bs_set_debug_flags(0x4) == INVALID
    assert lib.fp8bs_set_debug_flags(0) == OK


P = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


def _contig(**kw):
    args = dict(a=P, sa=P, sa_layout=0, ld_sa=0, b=P, sb=P, lay=P, d=P, out=0,
                m_sum=256, n=256, k=256, g=2)
    args.update(kw)
    return _binding.gemm_grouped_contiguous_raw(
        args["a"], args["sa"], args["sa_layout"], args["ld_sa"], args["b"], args["sb"],
        args["lay"], args["d"], args["out"], args["m_sum"], args["n"], args["k"], args["g"], 0)


def _masked(**kw):
    args = dict(a=P, sa=P, sa_layout=0, ld_sa=0, b=P, sb=P, mm=P, em=0, d=P, out=0,
                g=2, m_max=64, n=256, k=256)
    args.update(kw)
    return _binding.gemm_grouped_masked_raw(
        args["a"], args["sa"], args["sa_layout"], args["ld_sa"], args["b"], args["sb"],
        args["mm"], args["em"], args["d"], args["out"], args["g"], args["m_max"], args["n"],
        args["k"], 0)


@pytest.mark.parametrize("bad", [
    dict(a=0), dict(sa=0), dict(b=0), dict(sb=0), dict(lay=0), dict(d=0),
    dict(a=P + 8), dict(b=P + 4), dict(d=P + 2), dict(sa=P + 2), dict(lay=P + 1),
    dict(n=0), dict(n=200), dict(k=100), dict(k=-128), dict(g=0), dict(m_sum=-1),
    dict(out=2), dict(sa_layout=3),
    dict(sa_layout=1, ld_sa=255), dict(sa_layout=1, ld_sa=258), dict(sa_layout=1, ld_sa=256, sa=P + 4),
    dict(n=2 ** 30, g=4),
])
def test_contiguous_rejects(lib, bad):
    assert _contig(**bad) == INVALID


def test_contiguous_empty_is_noop(lib):
    assert _contig(m_sum=0, a=0, d=0) == OK
    assert _contig(m_sum=0, n=100) == INVALID


def test_rejected_and_empty_calls_launch_nothing(lib):
    n0 = fb.kernel_launches()
    assert _contig(k=100) == INVALID
    assert _contig(m_sum=0, a=0, d=0) == OK
    assert _masked(g=0) == INVALID
    assert fb.kernel_launches() == n0


@pytest.mark.parametrize("bad", [
    dict(mm=0), dict(a=0), dict(g=0), dict(g=1025), dict(m_max=-1), dict(n=128 + 64),
    dict(sa_layout=1, ld_sa=63), dict(sa_layout=1, ld_sa=66), dict(out=-1), dict(mm=P + 2),
])
def test_masked_rejects(lib, bad):
    assert _masked(**bad) == INVALID


def test_masked_empty_is_noop(lib):
    assert _masked(m_max=0, a=0) == OK


def test_scale_layout_from_strides():
    KB = 4
    sa_mk = torch.zeros(10, KB)
    assert _binding._sa_layout_2d(sa_mk, 10, KB) == (fb.SA_MK, KB)
    store = torch.zeros(KB, 12)
    assert _binding._sa_layout_2d(store[:, :10].t(), 10, KB) == (fb.SA_KM, 12)
    with pytest.raises(ValueError):
        _binding._sa_layout_2d(torch.zeros(10, 2 * KB)[:, ::2], 10, KB)
    m3 = torch.zeros(3, 5, KB)
    assert _binding._sa_layout_3d(m3, 3, 5, KB) == (fb.SA_MK, KB)
    s3 = torch.zeros(3, KB, 8)
    assert _binding._sa_layout_3d(s3[:, :, :5].transpose(1, 2), 3, 5, KB) == (fb.SA_KM, 8)


def test_wrappers_reject_host_tensors():
    # checked in the binding before any library call: a host tensor would reach the
    # kernel as an address it cannot use
    a = torch.zeros(256, 256, dtype=torch.uint8)
    sa = torch.ones(256, 2)
    b = torch.zeros(2, 256, 256, dtype=torch.uint8)
    sb = torch.ones(2, 2, 2)
    d = torch.zeros(256, 256, dtype=torch.bfloat16)
    lay = torch.zeros(256, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensors"):
        fb.gemm_grouped_contiguous(a, sa, b, sb, d, lay)
    with pytest.raises(ValueError, match="CUDA tensors"):
        fb.gemm_grouped_masked(a.view(1, 256, 256), sa.view(1, 256, 2), b[:1], sb[:1],
                               d.view(1, 256, 256), torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA tensors"):
        fb.gemm_grouped_contiguous_mxfp4(a[:, :128], torch.zeros(256, 8, dtype=torch.uint8),
                                         b[:, :, :128], torch.zeros(2, 256, 8, dtype=torch.uint8),
                                         d, lay)
    with pytest.raises(ValueError, match="CUDA tensors"):
        fb.gemm_grouped_contiguous_silu_mul_quant(a, sa, b, sb,
                                                  torch.zeros(256, 128, dtype=torch.uint8),
                                                  torch.ones(256, 1), lay)


def _noalloc(**kw):
    args = dict(a=P, sa=P, sa_layout=0, ld_sa=0, b=P, sb=P, lay=P, d=P, out=0,
                m_sum=256, n=256, k=256, g=2)
    args.update(kw)
    return _binding.gemm_grouped_contiguous_noalloc_raw(
        args["a"], args["sa"], args["sa_layout"], args["ld_sa"], args["b"], args["sb"],
        args["lay"], args["d"], args["out"], args["m_sum"], args["n"], args["k"], args["g"], 0)


@pytest.mark.parametrize("bad", [
    dict(n=200),                 # N a multiple of 128
    dict(d=P + 8),               # D 16-byte aligned like every entry point's
    dict(m_sum=524288 + 128),    # and at most 4096 row tiles (no workspace for a longer list)
    dict(g=1 << 15),             # and fewer than 2^15 groups (15-bit expert id of a list entry)
    dict(a=0), dict(k=100), dict(out=5),
])
def test_noalloc_rejects(lib, bad):
    assert _noalloc(**bad) == INVALID


def test_noalloc_empty_is_noop(lib):
    assert _noalloc(m_sum=0, a=0) == OK



def _fused(**kw):
    args = dict(a=P, sa=P, sa_layout=0, ld_sa=0, b=P, sb=P, lay=P, out=P, os=P, osl=0, ldo=0,
                m_sum=256, n=512, k=256, g=2)
    args.update(kw)
    return _binding.gemm_grouped_contiguous_silu_mul_quant_raw(
        args["a"], args["sa"], args["sa_layout"], args["ld_sa"], args["b"], args["sb"],
        args["lay"], args["out"], args["os"], args["osl"], args["ldo"], args["m_sum"], args["n"],
        args["k"], args["g"], 0)


def _fused_masked(**kw):
    args = dict(a=P, sa=P, sa_layout=0, ld_sa=0, b=P, sb=P, mm=P, out=P, os=P, osl=0, ldo=0,
                g=2, m_max=64, n=512, k=256)
    args.update(kw)
    return _binding.gemm_grouped_masked_silu_mul_quant_raw(
        args["a"], args["sa"], args["sa_layout"], args["ld_sa"], args["b"], args["sb"],
        args["mm"], 0, args["out"], args["os"], args["osl"], args["ldo"], args["g"],
        args["m_max"], args["n"], args["k"], 0)


@pytest.mark.parametrize("bad", [
    dict(n=384),                 # n/2 must be a multiple of 128
    dict(n=128),
    dict(out=P + 16),            # codes are stored 32 bytes at a time
    dict(os=0), dict(os=P + 2), dict(osl=2),
    dict(osl=1, ldo=255), dict(osl=1, ldo=258), dict(osl=1, ldo=256, os=P + 4),
    dict(m_sum=4194304 + 128),   # pair-list limit with the list in a device workspace
    dict(g=1 << 15),
    dict(a=0), dict(lay=0), dict(k=100), dict(sa_layout=5),
])
def test_fused_contiguous_rejects(lib, bad):
    assert _fused(**bad) == INVALID


@pytest.mark.parametrize("bad", [
    dict(n=384), dict(out=P + 16), dict(os=0), dict(osl=1, ldo=63), dict(osl=1, ldo=66),
    dict(mm=0), dict(g=0), dict(g=1025), dict(m_max=-1),
])
def test_fused_masked_rejects(lib, bad):
    assert _fused_masked(**bad) == INVALID


def test_fused_empty_is_noop(lib):
    assert _fused(m_sum=0, a=0, out=0, os=0) == OK
    assert _fused_masked(m_max=0, a=0, out=0, os=0) == OK
    assert _fused(m_sum=0, n=384) == INVALID


def _fp32s(**kw):
    args = dict(a=P, sa=P, sa_layout=0, ld_sa=0, b=P, sb=P, lay=P, d=P, out=0,
                m_sum=256, n=256, k=256, g=2)
    args.update(kw)
    return _binding.gemm_grouped_contiguous_fp32_scales_raw(
        args["a"], args["sa"], args["sa_layout"], args["ld_sa"], args["b"], args["sb"],
        args["lay"], args["d"], args["out"], args["m_sum"], args["n"], args["k"], args["g"], 0)


@pytest.mark.parametrize("bad", [
    dict(n=384),                 # the promotion kernel is a CTA-pair kernel: n % 256 == 0
    dict(d=P + 16),              # 32-byte output stores
    dict(m_sum=4194304 + 128), dict(g=1 << 15),
    dict(a=0), dict(sa=0), dict(lay=0), dict(k=100), dict(out=2), dict(sa_layout=1, ld_sa=255),
])
def test_fp32_scales_rejects(lib, bad):
    assert _fp32s(**bad) == INVALID


def test_fp32_scales_masked_rejects_and_empty(lib):
    def call(**kw):
        args = dict(a=P, sa=P, sa_layout=0, ld_sa=0, b=P, sb=P, mm=P, d=P, out=0, g=2, m_max=64,
                    n=256, k=256)
        args.update(kw)
        return _binding.gemm_grouped_masked_fp32_scales_raw(
            args["a"], args["sa"], args["sa_layout"], args["ld_sa"], args["b"], args["sb"],
            args["mm"], 0, args["d"], args["out"], args["g"], args["m_max"], args["n"],
            args["k"], 0)
    for bad in (dict(n=384), dict(d=P + 16), dict(mm=0), dict(g=0), dict(g=1025), dict(m_max=-1)):
        assert call(**bad) == INVALID, bad
    assert call(m_max=0, a=0) == OK
    assert _fp32s(m_sum=0, a=0, d=0) == OK


def _mx(**kw):
    args = dict(a=P, sa=P, b=P, sb=P, lay=P, d=P, out=0, m_sum=256, n=256, k=256, g=2)
    args.update(kw)
    return _binding.gemm_grouped_contiguous_mxfp4_raw(
        args["a"], args["sa"], args["b"], args["sb"], args["lay"], args["d"], args["out"],
        args["m_sum"], args["n"], args["k"], args["g"], 0)


@pytest.mark.parametrize("bad", [
    dict(k=128),                 # K blocks of 128 packed bytes: k % 256 == 0
    dict(n=384), dict(d=P + 16), dict(a=P + 8), dict(sa=P + 2), dict(sb=P + 1),
    dict(a=0), dict(sa=0), dict(lay=0), dict(out=3), dict(g=0),
    dict(m_sum=4194304 + 128),   # pair-list limit with the list in a device workspace
    dict(g=1 << 15),
])
def test_mxfp4_rejects(lib, bad):
    assert _mx(**bad) == INVALID


def test_mxfp4_masked_rejects_and_empty(lib):
    def call(**kw):
        args = dict(a=P, sa=P, b=P, sb=P, mm=P, d=P, out=0, g=2, m_max=64, n=256, k=256)
        args.update(kw)
        return _binding.gemm_grouped_masked_mxfp4_raw(
            args["a"], args["sa"], args["b"], args["sb"], args["mm"], 0, args["d"], args["out"],
            args["g"], args["m_max"], args["n"], args["k"], 0)
    for bad in (dict(k=128), dict(n=384), dict(mm=0), dict(d=P + 16), dict(g=1025)):
        assert call(**bad) == INVALID, bad
    assert call(m_max=0, a=0) == OK
    assert _mx(m_sum=0, a=0, d=0) == OK
