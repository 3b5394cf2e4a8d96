"""The E4M3 entry points take UE8M0 scales: fp32 powers of two whose exponent
field the tensor core applies ("Adds Grouped and Batched GEMM kernels with
blockscaling matching DeepGEMM API", DeepGEMM conformance details: scales
rounded with ceil_to_ue8m0 and applied by the matrix instruction).  A scale
of a stored row that is anything else -- not a power of two, zero, negative,
inf, NaN -- makes the call invalid and must set FP8BS_DEVERR_BAD_SCALE rather
than give silently truncated numbers.  Scales of rows that are not computed
(padding rows, rows past masked_m) are never read for a result and must not
raise it.  Rows that read only valid scales keep the parity tolerances.
Both activation-scale layouts are covered: row-major scales are checked by the
library's scale pre-pass, transposed ones inside the GEMM.
"""
import dataclasses

import numpy as np
import pytest
import torch

import fp8_block_scaled_gb300 as fb
import synth
from synth.inputs import SA_KM, SA_MK

from _parity import SENTINEL, all_rows, compare, out_torch_dtype, single_cta_kernel

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(p, sa, sb, single=False):
    """D bits [rows, N] and the device error word (read and cleared)."""
    d = torch.full((p.rows * p.N,), SENTINEL, dtype=torch.int16, device=DEV).view(out_torch_dtype(p))
    with single_cta_kernel(single):
        if p.variant == "contiguous":
            fb.gemm_grouped_contiguous(p.a, sa, p.b, sb, d.view(p.rows, p.N), p.grouped_layout)
        else:
            fb.gemm_grouped_masked(p.a, sa, p.b, sb, d.view(p.G, p.M_max, p.N), p.masked_m)
    torch.cuda.synchronize()
    flags = fb.device_error()
    return d.view(torch.int16).cpu().numpy().view(np.uint16).reshape(p.rows, p.N), flags


def _contiguous(n, seed, sa_layout=SA_MK):
    # expert 0: rows 0..199 (padding 200..255); expert 1: rows 256..405 (padding 406..511)
    return synth.make_problem("contiguous", 2, n, 512, [200, 150], sa_layout=sa_layout, seed=seed,
                              device=DEV)


def _sa_copy(p):
    """A copy of scale_a in p's stored layout, as its logical [rows, K/128] (masked:
    [G, M_max, K/128]) view: writes through the view land in the copy."""
    return dataclasses.replace(p, sa=p.sa.clone()).sa_mk_view()


LAYOUTS = [pytest.param(SA_MK, id="sa_mk"), pytest.param(SA_KM, id="sa_km")]


# the CTA-pair kernel (N=384: its last column tile is 128 wide) and, through the
# test hook, the single-CTA kernel
KERNELS = [pytest.param(512, False, id="pair"), pytest.param(384, False, id="pair_n384"),
           pytest.param(512, True, id="single_cta"), pytest.param(384, True, id="single_cta_n384")]


@pytest.mark.parametrize("sa_layout", LAYOUTS)
@pytest.mark.parametrize("n,single", KERNELS)
def test_bad_activation_scales_are_flagged(gg, n, single, sa_layout):
    p = _contiguous(n, seed=111, sa_layout=sa_layout)
    sa = _sa_copy(p)
    bad_rows = [10, 300, 301, 405]
    sa[10, 1] = 3.0              # not a power of two
    sa[300, 0] = -0.5            # negative
    sa[301, 2] = 0.0             # zero
    sa[405, 3] = float("inf")    # the last valid row of expert 1
    bits, flags = _run(p, sa, p.sb, single)
    assert flags & fb.DEVERR_BAD_SCALE, f"flags {flags:#x}"
    valid, untouched = all_rows(p)
    keep = np.setdiff1d(valid, bad_rows)
    compare(p, bits, keep, untouched, check_fp32=False)


@pytest.mark.parametrize("n,single", KERNELS)
def test_bad_weight_scale_is_flagged(gg, n, single):
    p = _contiguous(n, seed=112)
    sb = p.sb.clone()
    sb[1, 0, 1] = 1.25           # expert 1, columns 0..127, K block 1
    bits, flags = _run(p, p.sa_mk_view(), sb, single)
    assert flags & fb.DEVERR_BAD_SCALE, f"flags {flags:#x}"
    valid, untouched = all_rows(p)
    compare(p, bits, valid[valid < 256], untouched, check_fp32=False)  # expert 0 only


@pytest.mark.parametrize("sa_layout", LAYOUTS)
@pytest.mark.parametrize("n,single", KERNELS)
def test_scales_of_rows_not_computed_are_not_checked(gg, n, single, sa_layout):
    """Zero, NaN and non-power-of-two scales on padding rows (and on the ragged
    tail of the tile) leave the error word clear and the output bit-identical."""
    p = _contiguous(n, seed=113, sa_layout=sa_layout)
    ref, flags = _run(p, p.sa_mk_view(), p.sb, single)
    assert flags == 0
    sa = _sa_copy(p)
    sa[200:256] = 0.0
    sa[406:512, 0] = float("nan")
    sa[450, 2] = 3.0
    bits, flags = _run(p, sa, p.sb, single)
    assert flags == 0, f"flags {flags:#x}"
    assert np.array_equal(bits, ref)


@pytest.mark.parametrize("sa_layout", LAYOUTS)
@pytest.mark.parametrize("n", [512, 384])
def test_masked_rows_past_masked_m_are_not_checked(gg, n, sa_layout):
    p = synth.make_problem("masked", 2, n, 512, [70, 129], M_max=256, sa_layout=sa_layout,
                           seed=114, device=DEV)
    ref, flags = _run(p, p.sa_mk_view(), p.sb)
    assert flags == 0
    sa = _sa_copy(p)
    sa[0, 70:] = 0.0             # group 0 past masked_m
    sa[1, 129:, 1] = -2.0        # group 1 past masked_m
    bits, flags = _run(p, sa, p.sb)
    assert flags == 0, f"flags {flags:#x}"
    assert np.array_equal(bits, ref)
    sa[1, 128, 0] = 0.75         # group 1's last computed row
    bits, flags = _run(p, sa, p.sb)
    assert flags & fb.DEVERR_BAD_SCALE, f"flags {flags:#x}"
    valid, untouched = all_rows(p)
    keep = valid[valid != 256 + 128]
    compare(p, bits, keep, untouched, check_fp32=False)


@pytest.mark.parametrize("sa_layout", LAYOUTS)
def test_smallest_and_largest_ue8m0_scales_are_accepted(gg, sa_layout):
    """2^-127 (fp32 subnormal 0x00400000, UE8M0 code 0) and 2^127 (code 254)
    are UE8M0 values: no flag.  They change the results of their rows, which
    are not compared; every other row is."""
    p = _contiguous(512, seed=115, sa_layout=sa_layout)
    sa = _sa_copy(p)
    sa[5, 0] = float(np.ldexp(np.float32(1.0), -127))
    sa[6, 0] = float(np.ldexp(np.float32(1.0), 127))
    assert sa[5, 0:1].contiguous().view(torch.int32).item() == 0x00400000
    bits, flags = _run(p, sa, p.sb)
    assert flags == 0, f"flags {flags:#x}"
    valid, untouched = all_rows(p)
    compare(p, bits, np.setdiff1d(valid, [5, 6]), untouched, check_fp32=False)


@pytest.mark.parametrize("sa_layout", LAYOUTS)
def test_fused_epilogue_flags_bad_scales(gg, sa_layout):
    p = synth.make_problem("contiguous", 2, 512, 512, [200, 150], sa_layout=sa_layout, seed=116,
                           device=DEV)
    sa = _sa_copy(p)
    sa[20, 0] = 0.3
    q = torch.zeros((p.rows, p.N // 2), dtype=torch.uint8, device=DEV)
    s = torch.zeros((p.rows, p.N // 256), dtype=torch.float32, device=DEV)
    fb.gemm_grouped_contiguous_silu_mul_quant(p.a, sa, p.b, p.sb, q, s, p.grouped_layout)
    torch.cuda.synchronize()
    assert fb.device_error() & fb.DEVERR_BAD_SCALE
