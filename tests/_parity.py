"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
on a seeded problem and compare it with the CPU oracle row by row.

Tolerances (stated for the grouped block-scaled GEMM in fp32 accumulation
with bf16/f16 output):
  * calc_diff(D_gpu, D_oracle) <= 1e-5 over the compared valid rows;
  * per element |D_gpu - D_oracle| <= 2^-7 * |D_oracle| + 1e-2 * rms(D_oracle);
  * calc_diff(D_gpu, a_f32 @ b_f32^T) <= 1e-3 (the threshold and reference
    convention of the FlyDSL PR #433 page, section "DeepGEMM conformance
    details");
  * rows that must not be computed keep the sentinel bit pattern.
"""
from __future__ import annotations

import contextlib

import numpy as np
import torch

import fp8_block_scaled_gb300 as fb
import oracle
import synth

SENTINEL = 0x7FA5  # a NaN in both bf16 and f16
CALC_DIFF_ORACLE = 1e-5
CALC_DIFF_FP32 = 1e-3
# MXFP4 operands carry one mantissa bit: rounding each operand to E2M1 costs
# about 10% relative rms error, so calc_diff against the pre-quantisation fp32
# product is about 0.5 * (0.14)^2 ~= 0.01; the check allows 5x that.
CALC_DIFF_FP32_MX = 5e-2
REL_TOL = 2.0 ** -7
RMS_TOL = 1e-2


def out_torch_dtype(p):
    return torch.bfloat16 if p.out_dtype == synth.inputs.OUT_BF16 else torch.float16


def run_gpu(p, d=None, stream=None):
    """Run the problem (tensors already on the GPU) and return D as uint16 bits on the host,
    flattened to [rows, N]."""
    if p.variant == "contiguous":
        shape = (p.a.shape[0], p.N)
    else:
        shape = (p.G, p.M_max, p.N)
    if d is None:
        d = torch.full(shape, SENTINEL, dtype=torch.int16 if SENTINEL < 0x8000 else torch.int32,
                       device=p.a.device).view(out_torch_dtype(p))
    if p.is_mx:
        if p.variant == "contiguous":
            fb.gemm_grouped_contiguous_mxfp4(p.a, p.sa, p.b, p.sb, d, p.grouped_layout,
                                             stream=stream)
        else:
            fb.gemm_grouped_masked_mxfp4(p.a, p.sa, p.b, p.sb, d, p.masked_m, stream=stream)
        torch.cuda.synchronize()
        err = fb.device_error()
        assert err == 0, f"device error word {err:#x}"
        return d.view(torch.int16).reshape(-1, p.N).cpu().numpy().view(np.uint16)
    sa = p.sa_mk_view()
    promote = p.scale_kind == "fp32"   # arbitrary fp32 scales: the software-promotion kernel
    if p.variant == "contiguous":
        fn = fb.gemm_grouped_contiguous_fp32_scales if promote else fb.gemm_grouped_contiguous
        fn(p.a, sa, p.b, p.sb, d, p.grouped_layout, stream=stream)
    else:
        fn = fb.gemm_grouped_masked_fp32_scales if promote else fb.gemm_grouped_masked
        fn(p.a, sa, p.b, p.sb, d, p.masked_m, stream=stream)
    torch.cuda.synchronize()
    err = fb.device_error()
    assert err == 0, f"device error word {err:#x}"
    return d.view(torch.int16).reshape(-1, p.N).cpu().numpy().view(np.uint16)


def oracle_rows(p, rows):
    """Oracle fp64 accumulators for the listed flattened rows."""
    a = p.a.cpu().numpy()
    b = p.b.cpu().numpy()
    sa = p.sa.cpu().numpy()
    sb = p.sb.cpu().numpy()
    if p.is_mx:
        if p.variant == "contiguous":
            acc, valid, _ = oracle.mxfp4_contiguous(a, sa, b, sb, p.grouped_layout.cpu().numpy(),
                                                    rows=rows)
        else:
            acc, valid, _ = oracle.mxfp4_masked(a, sa, b, sb, p.masked_m.cpu().numpy(), rows=rows)
        return acc, valid
    if p.variant == "contiguous":
        acc, valid, _ = oracle.grouped_contiguous(a, sa, p.sa_layout, b, sb,
                                                  p.grouped_layout.cpu().numpy(), rows=rows,
                                                  ld_sa=p.ld_sa)
    else:
        acc, valid, _ = oracle.grouped_masked(a, sa, p.sa_layout, b, sb, p.masked_m.cpu().numpy(),
                                              rows=rows, ld_sa=p.ld_sa)
    return acc, valid


def fp32_reference_rows(p, rows):
    """a_f32 @ b_f32^T in fp64 for the listed valid rows (regenerated per group)."""
    out = np.empty((len(rows), p.N), dtype=np.float64)
    by_group = {}
    for i, r in enumerate(rows):
        g, m = p.group_of_row(int(r))
        assert g >= 0
        by_group.setdefault(g, []).append((i, m))
    for g, items in by_group.items():
        a32 = p.regen_a_f32(g)
        b32 = p.regen_b_f32(g).double().cpu()
        idx = torch.tensor([m for _, m in items], device=a32.device)
        prod = a32[idx].double().cpu() @ b32.T
        for j, (i, _) in enumerate(items):
            out[i] = prod[j].numpy()
    return out


def compare(p, bits, rows, untouched=(), check_fp32=True):
    """Assert the tolerances above for `rows` (flattened indices) of `bits`."""
    rows = np.asarray(rows, dtype=np.int64)
    acc, valid = oracle_rows(p, rows)
    assert valid.all(), "compare() takes valid rows only"
    got = oracle.bits_to_float(bits[rows], p.out_dtype)
    assert np.isfinite(got).all(), "non-finite output on a valid row"
    ref_bits = oracle.round_out(acc, p.out_dtype)
    ref = oracle.bits_to_float(ref_bits, p.out_dtype)
    cd = oracle.calc_diff(got, acc)
    assert cd <= CALC_DIFF_ORACLE, f"calc_diff vs oracle {cd:.3e}"
    rms = float(np.sqrt(np.mean(acc ** 2))) if acc.size else 0.0
    bound = REL_TOL * np.abs(acc) + RMS_TOL * rms
    err = np.abs(got - acc)
    assert (err <= bound).all(), f"max excess {(err - bound).max():.3e}"
    stats = {"calc_diff_oracle": cd, "exact_frac": float((ref_bits == bits[rows]).mean()),
             "rows": int(rows.size)}
    if check_fp32:
        ref32 = fp32_reference_rows(p, rows)
        cd32 = oracle.calc_diff(got, ref32)
        assert cd32 <= (CALC_DIFF_FP32_MX if p.is_mx else CALC_DIFF_FP32), \
            f"calc_diff vs fp32 {cd32:.3e}"
        stats["calc_diff_fp32"] = cd32
    untouched = np.asarray(untouched, dtype=np.int64)
    if untouched.size:
        assert (bits[untouched] == SENTINEL).all(), "a row that must not be written was written"
    return stats


def all_rows(p):
    """(valid rows, untouched rows) of a problem, flattened."""
    valid, untouched = [], []
    for r in range(p.rows):
        (valid if p.group_of_row(r)[0] >= 0 else untouched).append(r)
    return np.array(valid, np.int64), np.array(untouched, np.int64)


@contextlib.contextmanager
def single_cta_kernel(on=True):
    """Route the plain entry points to the single-CTA kernel (test hook) inside the block."""
    if on:
        fb.set_debug_flags(fb.DEBUG_SINGLE_CTA)
    try:
        yield
    finally:
        if on:
            fb.set_debug_flags(0)
