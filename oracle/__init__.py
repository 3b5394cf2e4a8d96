"""CPU oracle for the grouped FP8 (e4m3) block-scaled GEMM -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` leg of ``bench.py`` may import this package.  The CUDA
library in ``fp8_block_scaled_gb300`` never imports, links or calls it, and
the two share no code: this package wraps ``fp8bs_oracle.c`` (plain C, fp64)
through ctypes and adds nothing but argument marshalling.

What it computes follows "Adds Grouped and Batched GEMM kernels with
blockscaling matching DeepGEMM API" (FlyDSL PR #433), sections *Summary* and
*DeepGEMM conformance details*: for every valid row r of group g and every
column n,

    acc[r, n] = sum_kb sa[r, kb] * sb[g, n // 128, kb]
                       * sum_{k in block kb} e4m3(A[r, k]) * e4m3(B[g, n, k])

in fp64, then round-to-nearest-even to bf16 or f16.  Padding rows
(grouped_layout == -1) and rows at or beyond masked_m[g] produce no output.

Parity status of every function (see tests/test_oracle_pins.py):
  e4m3_decode       pinned: exhaustive vs torch.float8_e4m3fn conversion
  e4m3_encode       pinned: vs torch conversion on all in-range ties and samples
  ceil_to_ue8m0     pinned: closed-form properties, exhaustive powers of two +-1 ulp
  round_bf16/f16    pinned: vs torch fp32->bf16 and numpy fp64->f16
  contiguous/masked pinned: exact-rational brute force, integer matmul,
                    power-of-two scaling, masked==contiguous, group permutation,
                    pre-quantisation fp32 product within calc_diff 1e-3
  calc_diff         pinned: closed forms
  block_dot_exact   pinned: exact-rational brute force
  e2m1 / e8m0       pinned: the 16 E2M1 values derived by hand; E8M0 closed form
  mxfp4 GEMM        pinned: exact-rational brute force, integer matmul, power-of-two
                    scale exactness, masked == contiguous, nibble order
  silu_mul_quant    pinned: hand-derived golden blocks, SiLU closed forms and the
                    identity silu(x) - silu(-x) = x, quantiser invariants (power-of-two
                    scale, |h|/s <= 448, half-spacing error, sign), zero blocks

The fused gate/up epilogue (silu_mul_quant) follows "flydsl mxfp4 a4w4 MoE:
bring gemm1/gemm2 to parity with the HIP backend" (aiter PR #3828), section
*gemm1* (silu_mul of the gate and up halves), and requantises with the (1,128)
UE8M0 ceil quantiser of the FlyDSL PR #433 page, *DeepGEMM conformance details*.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

SA_MK = 0  # scale_a stored [rows, K/128]
SA_KM = 1  # scale_a stored transposed [K/128, ld_sa] (per group when masked)
OUT_BF16 = 0
OUT_F16 = 1

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build()
    lib = ctypes.CDLL(path)
    lib.fp8bs_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.fp8bs_oracle_e4m3_to_double.restype = ctypes.c_double
    lib.fp8bs_oracle_double_to_e4m3.argtypes = [ctypes.c_double]
    lib.fp8bs_oracle_double_to_e4m3.restype = ctypes.c_uint8
    lib.fp8bs_oracle_ceil_to_ue8m0.argtypes = [ctypes.c_double]
    lib.fp8bs_oracle_ceil_to_ue8m0.restype = ctypes.c_double
    lib.fp8bs_oracle_round_bf16.argtypes = [ctypes.c_double]
    lib.fp8bs_oracle_round_bf16.restype = ctypes.c_uint16
    lib.fp8bs_oracle_round_f16.argtypes = [ctypes.c_double]
    lib.fp8bs_oracle_round_f16.restype = ctypes.c_uint16
    lib.fp8bs_oracle_round_array.argtypes = [_P, _I64, ctypes.c_int, _P]
    lib.fp8bs_oracle_round_array.restype = None
    lib.fp8bs_oracle_contiguous.argtypes = [_P, _P, ctypes.c_int, _I64, _P, _P, _P,
                                            _I64, _I64, _I64, _I64, _P, _I64, _P, _P]
    lib.fp8bs_oracle_contiguous.restype = ctypes.c_int
    lib.fp8bs_oracle_masked.argtypes = [_P, _P, ctypes.c_int, _I64, _P, _P, _P,
                                        _I64, _I64, _I64, _I64, _P, _I64, _P, _P]
    lib.fp8bs_oracle_masked.restype = ctypes.c_int
    lib.fp8bs_oracle_calc_diff.argtypes = [_P, _P, _I64]
    lib.fp8bs_oracle_calc_diff.restype = ctypes.c_double
    lib.fp8bs_oracle_block_dot_exact.argtypes = [_P, _P]
    lib.fp8bs_oracle_block_dot_exact.restype = ctypes.c_double
    lib.fp8bs_oracle_silu_mul_quant.argtypes = [_P, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P]
    lib.fp8bs_oracle_silu_mul_quant.restype = ctypes.c_int
    lib.fp8bs_oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
    lib.fp8bs_oracle_e2m1_to_double.restype = ctypes.c_double
    lib.fp8bs_oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
    lib.fp8bs_oracle_e8m0_to_double.restype = ctypes.c_double
    lib.fp8bs_oracle_mxfp4_contiguous.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                                  _P, _I64, _P, _P]
    lib.fp8bs_oracle_mxfp4_contiguous.restype = ctypes.c_int
    lib.fp8bs_oracle_mxfp4_masked.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                              _P, _I64, _P, _P]
    lib.fp8bs_oracle_mxfp4_masked.restype = ctypes.c_int
    lib.fp8bs_oracle_max_threads.argtypes = []
    lib.fp8bs_oracle_max_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(x: np.ndarray):
    return x.ctypes.data_as(ctypes.c_void_p)


def _c(x, dtype):
    return np.ascontiguousarray(x, dtype=dtype)


def max_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all host cores)."""
    return int(_load().fp8bs_oracle_max_threads())


# ----------------------------------------------------------------- element codecs
def e4m3_decode(codes) -> np.ndarray:
    """E4M3 (OCP FN) byte codes -> fp64 values, decoded from the format definition."""
    lib = _load()
    codes = np.asarray(codes, dtype=np.uint8)
    flat = [lib.fp8bs_oracle_e4m3_to_double(int(c)) for c in codes.reshape(-1)]
    return np.array(flat, dtype=np.float64).reshape(codes.shape)


def e4m3_table() -> np.ndarray:
    """The 256 decoded E4M3 values, index = byte code."""
    return e4m3_decode(np.arange(256, dtype=np.uint8))


def e4m3_encode(x) -> np.ndarray:
    """fp64 -> E4M3 codes, round-to-nearest-even, saturating at +-448."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    flat = [lib.fp8bs_oracle_double_to_e4m3(float(v)) for v in x.reshape(-1)]
    return np.array(flat, dtype=np.uint8).reshape(x.shape)


def ceil_to_ue8m0(t) -> np.ndarray:
    """Smallest power of two >= t, for t > 0 (fp64 in, fp64 out)."""
    lib = _load()
    t = np.asarray(t, dtype=np.float64)
    flat = [lib.fp8bs_oracle_ceil_to_ue8m0(float(v)) for v in t.reshape(-1)]
    return np.array(flat, dtype=np.float64).reshape(t.shape)


def round_out(x, out_dtype: int) -> np.ndarray:
    """fp64 -> bf16 (out_dtype 0) or f16 (1) bit patterns, round-to-nearest-even."""
    lib = _load()
    x = _c(x, np.float64)
    bits = np.empty(x.shape, dtype=np.uint16)
    lib.fp8bs_oracle_round_array(_ptr(x), x.size, int(out_dtype), _ptr(bits))
    return bits


def bits_to_float(bits, out_dtype: int) -> np.ndarray:
    """bf16/f16 bit patterns -> fp64 values (exact widening)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if out_dtype == OUT_F16:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def calc_diff(x, y) -> float:
    """1 - 2*sum(xy) / (sum(x^2) + sum(y^2)) in fp64 (0 when both are zero)."""
    x = _c(x, np.float64).reshape(-1)
    y = _c(y, np.float64).reshape(-1)
    if x.size != y.size:
        raise ValueError("calc_diff: size mismatch")
    return float(_load().fp8bs_oracle_calc_diff(_ptr(x), _ptr(y), x.size))


def block_dot_exact(x_codes, y_codes) -> float:
    """Exact 128-element E4M3 dot product via int64 arithmetic in units of 2^-18."""
    x = _c(x_codes, np.uint8).reshape(-1)
    y = _c(y_codes, np.uint8).reshape(-1)
    if x.size != 128 or y.size != 128:
        raise ValueError("block_dot_exact takes two 128-element blocks")
    return float(_load().fp8bs_oracle_block_dot_exact(_ptr(x), _ptr(y)))


# ----------------------------------------------------------------- grouped GEMM
def grouped_contiguous(a_codes, scale_a, sa_layout, b_codes, scale_b, grouped_layout,
                       rows=None, ld_sa=None):
    """Contiguous grouped GEMM for the listed rows (default: all rows).

    a_codes  uint8 [M_sum, K]    e4m3 codes
    scale_a  fp32  [M_sum, K/128] (SA_MK) or [K/128, ld_sa] (SA_KM)
    b_codes  uint8 [G, N, K]
    scale_b  fp32  [G, N/128, K/128]
    grouped_layout int32 [M_sum], -1 = padding row

    Returns (acc fp64 [len(rows), N], valid bool [len(rows)], rows int64).
    """
    a = _c(a_codes, np.uint8)
    b = _c(b_codes, np.uint8)
    sa = _c(scale_a, np.float32)
    sb = _c(scale_b, np.float32)
    lay = _c(grouped_layout, np.int32)
    m_sum, k = a.shape
    g_count, n, kb = b.shape
    if kb != k:
        raise ValueError("K mismatch between A and B")
    if ld_sa is None:
        ld_sa = sa.shape[1] if sa_layout == SA_KM else k // 128
    rows = np.arange(m_sum, dtype=np.int64) if rows is None else _c(rows, np.int64)
    acc = np.empty((rows.size, n), dtype=np.float64)
    valid = np.empty(rows.size, dtype=np.uint8)
    rc = _load().fp8bs_oracle_contiguous(_ptr(a), _ptr(sa), int(sa_layout), int(ld_sa),
                                         _ptr(b), _ptr(sb), _ptr(lay), m_sum, n, k, g_count,
                                         _ptr(rows), rows.size, _ptr(acc), _ptr(valid))
    if rc != 0:
        raise ValueError("oracle: invalid arguments")
    return acc, valid.astype(bool), rows


def grouped_masked(a_codes, scale_a, sa_layout, b_codes, scale_b, masked_m,
                   rows=None, ld_sa=None):
    """Masked grouped GEMM for the listed flattened rows g*M_max + m (default: all).

    a_codes  uint8 [G, M_max, K]
    scale_a  fp32  [G, M_max, K/128] (SA_MK) or [G, K/128, ld_sa] (SA_KM)
    b_codes  uint8 [G, N, K];  scale_b fp32 [G, N/128, K/128]
    masked_m int32 [G]
    """
    a = _c(a_codes, np.uint8)
    b = _c(b_codes, np.uint8)
    sa = _c(scale_a, np.float32)
    sb = _c(scale_b, np.float32)
    mm = _c(masked_m, np.int32)
    g_count, m_max, k = a.shape
    _, n, _ = b.shape
    if ld_sa is None:
        ld_sa = sa.shape[2] if sa_layout == SA_KM else k // 128
    rows = (np.arange(g_count * m_max, dtype=np.int64) if rows is None
            else _c(rows, np.int64))
    acc = np.empty((rows.size, n), dtype=np.float64)
    valid = np.empty(rows.size, dtype=np.uint8)
    rc = _load().fp8bs_oracle_masked(_ptr(a), _ptr(sa), int(sa_layout), int(ld_sa),
                                     _ptr(b), _ptr(sb), _ptr(mm), g_count, m_max, n, k,
                                     _ptr(rows), rows.size, _ptr(acc), _ptr(valid))
    if rc != 0:
        raise ValueError("oracle: invalid arguments")
    return acc, valid.astype(bool), rows


# ----------------------------------------------------------------- fused gate/up epilogue
def silu_mul_quant(acc_gate_up):
    """SiLU(gate) * up of a [rows, 2I] accumulator (gate = columns [0, I), up =
    [I, 2I)), requantised per (1,128) block to E4M3 with UE8M0 ceil scales.

    Returns a dict of numpy arrays:
      h        fp64  [rows, I]      the exact activation
      q        uint8 [rows, I]      E4M3 codes
      s        fp32  [rows, I/128]  power-of-two scales
      margin   fp64  [rows, I]      relative distance of fl32(h)/s to the nearest
                                    E4M3 rounding boundary
      tmargin  fp64  [rows, I/128]  relative distance of amax/448 to the nearest
                                    power of two
    """
    acc = _c(acc_gate_up, np.float64)
    rows, n2 = acc.shape
    if n2 % 256:
        raise ValueError("silu_mul_quant: the accumulator needs 2I columns, I % 128 == 0")
    i_out = n2 // 2
    h = np.empty((rows, i_out), dtype=np.float64)
    q = np.empty((rows, i_out), dtype=np.uint8)
    s = np.empty((rows, i_out // 128), dtype=np.float32)
    margin = np.empty((rows, i_out), dtype=np.float64)
    tmargin = np.empty((rows, i_out // 128), dtype=np.float64)
    gate = np.ascontiguousarray(acc[:, :i_out])
    up = np.ascontiguousarray(acc[:, i_out:])
    rc = _load().fp8bs_oracle_silu_mul_quant(_ptr(gate), _ptr(up), rows, i_out, i_out,
                                             _ptr(h), _ptr(q), _ptr(s), _ptr(margin),
                                             _ptr(tmargin))
    if rc != 0:
        raise ValueError("oracle: invalid arguments")
    return {"h": h, "q": q, "s": s, "margin": margin, "tmargin": tmargin}


# ----------------------------------------------------------------- MXFP4 grouped GEMM
def e2m1_decode(codes) -> np.ndarray:
    """E2M1 4-bit codes (0..15) -> fp64 values, from the format definition."""
    lib = _load()
    codes = np.asarray(codes, dtype=np.uint8)
    flat = [lib.fp8bs_oracle_e2m1_to_double(int(c) & 0xF) for c in codes.reshape(-1)]
    return np.array(flat, dtype=np.float64).reshape(codes.shape)


def e8m0_decode(codes) -> np.ndarray:
    """E8M0 scale bytes -> 2^(e - 127) (NaN for 255)."""
    lib = _load()
    codes = np.asarray(codes, dtype=np.uint8)
    flat = [lib.fp8bs_oracle_e8m0_to_double(int(c)) for c in codes.reshape(-1)]
    return np.array(flat, dtype=np.float64).reshape(codes.shape)


def mxfp4_contiguous(a_packed, scale_a, b_packed, scale_b, grouped_layout, rows=None):
    """Contiguous MXFP4 grouped GEMM for the listed rows (default: all).

    a_packed uint8 [M_sum, K/2] (element 2i in the low nibble of byte i)
    scale_a  uint8 [M_sum, K/32] E8M0;  b_packed uint8 [G, N, K/2];
    scale_b  uint8 [G, N, K/32];  grouped_layout int32 [M_sum], -1 = padding.
    Returns (acc fp64 [len(rows), N], valid bool, rows).
    """
    a = _c(a_packed, np.uint8)
    b = _c(b_packed, np.uint8)
    sa = _c(scale_a, np.uint8)
    sb = _c(scale_b, np.uint8)
    lay = _c(grouped_layout, np.int32)
    m_sum, kh = a.shape
    g_count, n, _ = b.shape
    rows = np.arange(m_sum, dtype=np.int64) if rows is None else _c(rows, np.int64)
    acc = np.empty((rows.size, n), dtype=np.float64)
    valid = np.empty(rows.size, dtype=np.uint8)
    rc = _load().fp8bs_oracle_mxfp4_contiguous(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(lay),
                                               m_sum, n, 2 * kh, g_count, _ptr(rows), rows.size,
                                               _ptr(acc), _ptr(valid))
    if rc != 0:
        raise ValueError("oracle: invalid arguments")
    return acc, valid.astype(bool), rows


def mxfp4_masked(a_packed, scale_a, b_packed, scale_b, masked_m, rows=None):
    """Masked MXFP4 grouped GEMM: a_packed [G, M_max, K/2], scale_a [G, M_max, K/32]."""
    a = _c(a_packed, np.uint8)
    b = _c(b_packed, np.uint8)
    sa = _c(scale_a, np.uint8)
    sb = _c(scale_b, np.uint8)
    mm = _c(masked_m, np.int32)
    g_count, m_max, kh = a.shape
    _, n, _ = b.shape
    rows = (np.arange(g_count * m_max, dtype=np.int64) if rows is None
            else _c(rows, np.int64))
    acc = np.empty((rows.size, n), dtype=np.float64)
    valid = np.empty(rows.size, dtype=np.uint8)
    rc = _load().fp8bs_oracle_mxfp4_masked(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(mm),
                                           g_count, m_max, n, 2 * kh, _ptr(rows), rows.size,
                                           _ptr(acc), _ptr(valid))
    if rc != 0:
        raise ValueError("oracle: invalid arguments")
    return acc, valid.astype(bool), rows
