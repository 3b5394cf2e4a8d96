"""ctypes binding of libfp8bs.so (argument marshalling only).

Every tensor stays on the GPU; the library receives raw device pointers,
sizes and the current CUDA stream.  There is no CPU fallback: if the library
cannot be built or loaded, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64

SA_MK = 0
SA_KM = 1
OUT_BF16 = 0
OUT_F16 = 1
DEVERR_TIMEOUT = 0x1
DEVERR_MASKED_M = 0x2
DEVERR_MIXED_TILE = 0x4
DEVERR_BAD_GROUP = 0x8
DEVERR_BAD_SCALE = 0x10

# every symbol include/fp8bs.h declares
EXPORTS = ("gemm_grouped_contiguous", "gemm_grouped_masked", "gemm_grouped_contiguous_noalloc",
           "gemm_grouped_contiguous_silu_mul_quant", "gemm_grouped_masked_silu_mul_quant",
           "gemm_grouped_contiguous_fp32_scales", "gemm_grouped_masked_fp32_scales",
           "gemm_grouped_contiguous_mxfp4", "gemm_grouped_masked_mxfp4",
           "fp8bs_device_error", "fp8bs_status_string", "fp8bs_clear_cache", "fp8bs_abi_version",
           "fp8bs_set_debug_flags", "fp8bs_kernel_launches")

_lib = None
_lock = threading.Lock()


class Fp8bsError(RuntimeError):
    """A non-zero status from the C ABI."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


def lib_path() -> str:
    return _build.LIB


def load(auto_build: bool = True) -> ctypes.CDLL:
    """Load the CUDA library (building it in-tree with nvcc when missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if auto_build and _build.is_stale():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise ImportError(f"fp8_block_scaled_gb300: CUDA library not built ({_build.LIB}); "
                              "run fp8_block_scaled_gb300.build.build()")
        lib = ctypes.CDLL(_build.LIB)
        lib.gemm_grouped_contiguous.argtypes = [_P, _P, _I, _I64, _P, _P, _P, _P, _I,
                                                _I64, _I64, _I64, _I64, _P]
        lib.gemm_grouped_contiguous.restype = _I
        lib.gemm_grouped_masked.argtypes = [_P, _P, _I, _I64, _P, _P, _P, _I64, _P, _I,
                                            _I64, _I64, _I64, _I64, _P]
        lib.gemm_grouped_masked.restype = _I
        lib.gemm_grouped_contiguous_noalloc.argtypes = [_P, _P, _I, _I64, _P, _P, _P, _P, _I,
                                                        _I64, _I64, _I64, _I64, _P]
        lib.gemm_grouped_contiguous_noalloc.restype = _I
        lib.gemm_grouped_contiguous_silu_mul_quant.argtypes = [_P, _P, _I, _I64, _P, _P, _P, _P, _P,
                                                               _I, _I64, _I64, _I64, _I64, _I64, _P]
        lib.gemm_grouped_contiguous_silu_mul_quant.restype = _I
        lib.gemm_grouped_masked_silu_mul_quant.argtypes = [_P, _P, _I, _I64, _P, _P, _P, _I64, _P,
                                                           _P, _I, _I64, _I64, _I64, _I64, _I64, _P]
        lib.gemm_grouped_masked_silu_mul_quant.restype = _I
        lib.gemm_grouped_contiguous_fp32_scales.argtypes = lib.gemm_grouped_contiguous.argtypes
        lib.gemm_grouped_contiguous_fp32_scales.restype = _I
        lib.gemm_grouped_masked_fp32_scales.argtypes = lib.gemm_grouped_masked.argtypes
        lib.gemm_grouped_masked_fp32_scales.restype = _I
        lib.gemm_grouped_contiguous_mxfp4.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64,
                                                      _I64, _P]
        lib.gemm_grouped_contiguous_mxfp4.restype = _I
        lib.gemm_grouped_masked_mxfp4.argtypes = [_P, _P, _P, _P, _P, _I64, _P, _I, _I64, _I64,
                                                  _I64, _I64, _P]
        lib.gemm_grouped_masked_mxfp4.restype = _I
        lib.fp8bs_device_error.argtypes = [_I, ctypes.POINTER(ctypes.c_uint32)]
        lib.fp8bs_device_error.restype = _I
        lib.fp8bs_status_string.argtypes = [_I]
        lib.fp8bs_status_string.restype = ctypes.c_char_p
        lib.fp8bs_clear_cache.argtypes = []
        lib.fp8bs_clear_cache.restype = _I
        lib.fp8bs_set_debug_flags.argtypes = [ctypes.c_uint32]
        lib.fp8bs_set_debug_flags.restype = _I
        lib.fp8bs_abi_version.argtypes = []
        lib.fp8bs_abi_version.restype = _I
        lib.fp8bs_kernel_launches.argtypes = []
        lib.fp8bs_kernel_launches.restype = ctypes.c_uint64
        _lib = lib
        return lib


def status_string(status: int) -> str:
    if _lib is None:
        return "?"
    return _lib.fp8bs_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != 0:
        raise Fp8bsError(status, what)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _out_code(d: torch.Tensor) -> int:
    if d.dtype == torch.bfloat16:
        return OUT_BF16
    if d.dtype == torch.float16:
        return OUT_F16
    raise TypeError("output must be bfloat16 or float16")


def _fp8_ptr(t: torch.Tensor, name: str) -> int:
    if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError(f"{name} must be float8_e4m3fn (or its uint8 codes)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _contig_ptr(t: torch.Tensor, name: str) -> int:
    # no silent .contiguous() copy: a temporary could be freed and its memory
    # reused on torch's current stream while the kernel still reads it on another
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _device_of(*tensors, stream=None) -> torch.device:
    """The one CUDA device holding every tensor (and the given torch stream).  The
    library launches on the calling thread's current device, so a call with tensors
    of another device (or of the host) would hand the kernel addresses it cannot use."""
    dev = None
    for t in tensors:
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"all tensors must be on one device ({dev} and {t.device} given)")
    sdev = getattr(stream, "device", None)
    if isinstance(sdev, torch.device) and sdev != dev:
        raise ValueError(f"stream is on {sdev}, the tensors on {dev}")
    return dev


def _sa_layout_2d(sa: torch.Tensor, rows: int, kb: int):
    """(layout, ld) of a logical [rows, K/128] scale tensor from its strides."""
    if sa.dtype != torch.float32 or sa.shape != (rows, kb):
        raise ValueError(f"scale_a must be fp32 [{rows}, {kb}], got {tuple(sa.shape)} {sa.dtype}")
    s0, s1 = sa.stride()
    if s1 == 1 and (s0 == kb or rows == 1):
        return SA_MK, kb
    if s0 == 1:
        return SA_KM, s1
    raise ValueError("scale_a must be row-major [M, K/128] or a transposed view of [K/128, ld]")


def _sa_layout_3d(sa: torch.Tensor, G: int, m_max: int, kb: int):
    if sa.dtype != torch.float32 or sa.shape != (G, m_max, kb):
        raise ValueError(f"scale_a must be fp32 [{G}, {m_max}, {kb}], got {tuple(sa.shape)}")
    s0, s1, s2 = sa.stride()
    if s2 == 1 and s1 == kb and s0 == m_max * kb:
        return SA_MK, kb
    if s1 == 1 and s0 == kb * s2:
        return SA_KM, s2
    raise ValueError("scale_a must be [G, M_max, K/128] row-major or a transposed view of "
                     "[G, K/128, ld]")


def gemm_grouped_contiguous_raw(a_ptr, sa_ptr, sa_layout, ld_sa, b_ptr, sb_ptr, layout_ptr,
                                d_ptr, out_dtype, m_sum, n, k, num_groups, stream=None) -> int:
    """Direct C-ABI call with raw device pointers; returns the status code."""
    lib = load()
    return lib.gemm_grouped_contiguous(a_ptr, sa_ptr, int(sa_layout), int(ld_sa), b_ptr, sb_ptr,
                                       layout_ptr, d_ptr, int(out_dtype), int(m_sum), int(n),
                                       int(k), int(num_groups), ctypes.c_void_p(_stream_handle(stream)))


def gemm_grouped_contiguous_noalloc_raw(a_ptr, sa_ptr, sa_layout, ld_sa, b_ptr, sb_ptr,
                                        layout_ptr, d_ptr, out_dtype, m_sum, n, k, num_groups,
                                        stream=None) -> int:
    """C-ABI call of the variant that allocates no device memory (raw pointers)."""
    lib = load()
    return lib.gemm_grouped_contiguous_noalloc(
        a_ptr, sa_ptr, int(sa_layout), int(ld_sa), b_ptr, sb_ptr, layout_ptr, d_ptr,
        int(out_dtype), int(m_sum), int(n), int(k), int(num_groups),
        ctypes.c_void_p(_stream_handle(stream)))


def gemm_grouped_masked_raw(a_ptr, sa_ptr, sa_layout, ld_sa, b_ptr, sb_ptr, masked_m_ptr,
                            expected_m, d_ptr, out_dtype, num_groups, m_max, n, k,
                            stream=None) -> int:
    lib = load()
    return lib.gemm_grouped_masked(a_ptr, sa_ptr, int(sa_layout), int(ld_sa), b_ptr, sb_ptr,
                                   masked_m_ptr, int(expected_m), d_ptr, int(out_dtype),
                                   int(num_groups), int(m_max), int(n), int(k),
                                   ctypes.c_void_p(_stream_handle(stream)))


def gemm_grouped_contiguous_fp32_scales_raw(a_ptr, sa_ptr, sa_layout, ld_sa, b_ptr, sb_ptr,
                                            layout_ptr, d_ptr, out_dtype, m_sum, n, k,
                                            num_groups, stream=None) -> int:
    lib = load()
    return lib.gemm_grouped_contiguous_fp32_scales(
        a_ptr, sa_ptr, int(sa_layout), int(ld_sa), b_ptr, sb_ptr, layout_ptr, d_ptr,
        int(out_dtype), int(m_sum), int(n), int(k), int(num_groups),
        ctypes.c_void_p(_stream_handle(stream)))


def gemm_grouped_masked_fp32_scales_raw(a_ptr, sa_ptr, sa_layout, ld_sa, b_ptr, sb_ptr,
                                        masked_m_ptr, expected_m, d_ptr, out_dtype, num_groups,
                                        m_max, n, k, stream=None) -> int:
    lib = load()
    return lib.gemm_grouped_masked_fp32_scales(
        a_ptr, sa_ptr, int(sa_layout), int(ld_sa), b_ptr, sb_ptr, masked_m_ptr, int(expected_m),
        d_ptr, int(out_dtype), int(num_groups), int(m_max), int(n), int(k),
        ctypes.c_void_p(_stream_handle(stream)))


def gemm_grouped_contiguous_fp32_scales(a, scale_a, b, scale_b, d, grouped_layout, *,
                                        stream=None):
    """As gemm_grouped_contiguous, with arbitrary fp32 block scales (software promotion)."""
    return gemm_grouped_contiguous(a, scale_a, b, scale_b, d, grouped_layout, stream=stream,
                                   _raw=gemm_grouped_contiguous_fp32_scales_raw)


def gemm_grouped_masked_fp32_scales(a, scale_a, b, scale_b, d, masked_m, expected_m: int = 0, *,
                                    stream=None):
    """As gemm_grouped_masked, with arbitrary fp32 block scales (software promotion)."""
    return gemm_grouped_masked(a, scale_a, b, scale_b, d, masked_m, expected_m, stream=stream,
                               _raw=gemm_grouped_masked_fp32_scales_raw)


def gemm_grouped_contiguous(a, scale_a, b, scale_b, d, grouped_layout, *, stream=None,
                            _raw=None):
    """D = grouped FP8 block-scaled GEMM, contiguous variant (see include/fp8bs.h).

    a [M_sum, K] e4m3; scale_a logical [M_sum, K/128] fp32 (row-major, or a
    transposed view of a [K/128, ld] buffer); b [G, N, K] e4m3; scale_b
    [G, N/128, K/128] fp32; d [M_sum, N] bf16/f16; grouped_layout [M_sum]
    int32 with -1 for padding rows.  Rows marked -1 are not written.
    """
    m_sum, k = a.shape
    G, n, kb_ = b.shape
    if kb_ != k or d.shape != (m_sum, n) or grouped_layout.shape != (m_sum,):
        raise ValueError("shape mismatch")
    if scale_b.shape != (G, n // 128, k // 128) or scale_b.dtype != torch.float32:
        raise ValueError("scale_b must be fp32 [G, N/128, K/128]")
    if grouped_layout.dtype != torch.int32 or not d.is_contiguous():
        raise ValueError("grouped_layout must be int32, d contiguous")
    dev = _device_of(a, scale_a, b, scale_b, d, grouped_layout, stream=stream)
    layout, ld = _sa_layout_2d(scale_a, m_sum, k // 128)
    raw = _raw or gemm_grouped_contiguous_raw
    with torch.cuda.device(dev):
        st = raw(_fp8_ptr(a, "a"), scale_a.data_ptr(), layout, ld, _fp8_ptr(b, "b"),
                 _contig_ptr(scale_b, "scale_b"), _contig_ptr(grouped_layout, "grouped_layout"),
                 d.data_ptr(), _out_code(d), m_sum, n, k, G, stream)
    _check(st, raw.__name__[:-4])
    return d


def gemm_grouped_masked(a, scale_a, b, scale_b, d, masked_m, expected_m: int = 0, *,
                        stream=None, _raw=None):
    """D = grouped FP8 block-scaled GEMM, masked variant (see include/fp8bs.h).

    a [G, M_max, K] e4m3; scale_a logical [G, M_max, K/128] fp32 (row-major,
    or a transposed view of a [G, K/128, ld] buffer); b [G, N, K]; scale_b
    [G, N/128, K/128]; d [G, M_max, N]; masked_m [G] int32 on the device.
    Rows m >= masked_m[g] are not written.
    """
    G, m_max, k = a.shape
    Gb, n, kb_ = b.shape
    if Gb != G or kb_ != k or d.shape != (G, m_max, n) or masked_m.shape != (G,):
        raise ValueError("shape mismatch")
    if scale_b.shape != (G, n // 128, k // 128) or scale_b.dtype != torch.float32:
        raise ValueError("scale_b must be fp32 [G, N/128, K/128]")
    if masked_m.dtype != torch.int32 or not d.is_contiguous():
        raise ValueError("masked_m must be int32, d contiguous")
    dev = _device_of(a, scale_a, b, scale_b, d, masked_m, stream=stream)
    layout, ld = _sa_layout_3d(scale_a, G, m_max, k // 128)
    raw = _raw or gemm_grouped_masked_raw
    with torch.cuda.device(dev):
        st = raw(_fp8_ptr(a, "a"), scale_a.data_ptr(), layout, ld, _fp8_ptr(b, "b"),
                 _contig_ptr(scale_b, "scale_b"), _contig_ptr(masked_m, "masked_m"), expected_m,
                 d.data_ptr(), _out_code(d), G, m_max, n, k, stream)
    _check(st, raw.__name__[:-4])
    return d


def gemm_grouped_contiguous_silu_mul_quant_raw(a_ptr, sa_ptr, sa_layout, ld_sa, b_ptr, sb_ptr,
                                               layout_ptr, out_ptr, out_scale_ptr,
                                               out_scale_layout, ld_out_scale, m_sum, n, k,
                                               num_groups, stream=None) -> int:
    lib = load()
    return lib.gemm_grouped_contiguous_silu_mul_quant(
        a_ptr, sa_ptr, int(sa_layout), int(ld_sa), b_ptr, sb_ptr, layout_ptr, out_ptr,
        out_scale_ptr, int(out_scale_layout), int(ld_out_scale), int(m_sum), int(n), int(k),
        int(num_groups), ctypes.c_void_p(_stream_handle(stream)))


def gemm_grouped_masked_silu_mul_quant_raw(a_ptr, sa_ptr, sa_layout, ld_sa, b_ptr, sb_ptr,
                                           masked_m_ptr, expected_m, out_ptr, out_scale_ptr,
                                           out_scale_layout, ld_out_scale, num_groups, m_max, n,
                                           k, stream=None) -> int:
    lib = load()
    return lib.gemm_grouped_masked_silu_mul_quant(
        a_ptr, sa_ptr, int(sa_layout), int(ld_sa), b_ptr, sb_ptr, masked_m_ptr, int(expected_m),
        out_ptr, out_scale_ptr, int(out_scale_layout), int(ld_out_scale), int(num_groups),
        int(m_max), int(n), int(k), ctypes.c_void_p(_stream_handle(stream)))


def _check_out(out, out_scale, lead, n):
    if out.dtype not in (torch.float8_e4m3fn, torch.uint8) or not out.is_contiguous():
        raise TypeError("out must be a contiguous float8_e4m3fn (or uint8) tensor")
    if out.shape != tuple(lead) + (n // 2,):
        raise ValueError(f"out must be {tuple(lead) + (n // 2,)}")
    if out_scale.dtype != torch.float32:
        raise TypeError("out_scale must be fp32")


def gemm_grouped_contiguous_silu_mul_quant(a, scale_a, b, scale_b, out, out_scale,
                                           grouped_layout, *, stream=None):
    """Fused gate/up GEMM + SiLU(gate) * up + (1,128) E4M3 requantisation (include/fp8bs.h).

    b [G, N, K] holds the gate rows [0, N/2) and the up rows [N/2, N) of each
    expert.  out [M_sum, N/2] receives E4M3 codes; out_scale is the logical
    [M_sum, N/256] fp32 scale tensor (row-major, or a transposed view of a
    [N/256, ld] buffer) -- the activation operand of the down projection.
    Rows marked -1 are not written.
    """
    m_sum, k = a.shape
    G, n, kb_ = b.shape
    if kb_ != k or grouped_layout.shape != (m_sum,) or grouped_layout.dtype != torch.int32:
        raise ValueError("shape mismatch")
    if scale_b.shape != (G, n // 128, k // 128) or scale_b.dtype != torch.float32:
        raise ValueError("scale_b must be fp32 [G, N/128, K/128]")
    _check_out(out, out_scale, (m_sum,), n)
    dev = _device_of(a, scale_a, b, scale_b, out, out_scale, grouped_layout, stream=stream)
    layout, ld = _sa_layout_2d(scale_a, m_sum, k // 128)
    olayout, old = _sa_layout_2d(out_scale, m_sum, n // 256)
    with torch.cuda.device(dev):
        st = gemm_grouped_contiguous_silu_mul_quant_raw(
            _fp8_ptr(a, "a"), scale_a.data_ptr(), layout, ld, _fp8_ptr(b, "b"),
            _contig_ptr(scale_b, "scale_b"), _contig_ptr(grouped_layout, "grouped_layout"),
            out.data_ptr(), out_scale.data_ptr(), olayout, old, m_sum, n, k, G, stream)
    _check(st, "gemm_grouped_contiguous_silu_mul_quant")
    return out, out_scale


def gemm_grouped_masked_silu_mul_quant(a, scale_a, b, scale_b, out, out_scale, masked_m,
                                       expected_m: int = 0, *, stream=None):
    """Masked variant: a [G, M_max, K]; out [G, M_max, N/2]; out_scale logical
    [G, M_max, N/256] (row-major or a transposed view of [G, N/256, ld])."""
    G, m_max, k = a.shape
    Gb, n, kb_ = b.shape
    if Gb != G or kb_ != k or masked_m.shape != (G,) or masked_m.dtype != torch.int32:
        raise ValueError("shape mismatch")
    if scale_b.shape != (G, n // 128, k // 128) or scale_b.dtype != torch.float32:
        raise ValueError("scale_b must be fp32 [G, N/128, K/128]")
    _check_out(out, out_scale, (G, m_max), n)
    dev = _device_of(a, scale_a, b, scale_b, out, out_scale, masked_m, stream=stream)
    layout, ld = _sa_layout_3d(scale_a, G, m_max, k // 128)
    olayout, old = _sa_layout_3d(out_scale, G, m_max, n // 256)
    with torch.cuda.device(dev):
        st = gemm_grouped_masked_silu_mul_quant_raw(
            _fp8_ptr(a, "a"), scale_a.data_ptr(), layout, ld, _fp8_ptr(b, "b"),
            _contig_ptr(scale_b, "scale_b"), _contig_ptr(masked_m, "masked_m"), expected_m,
            out.data_ptr(), out_scale.data_ptr(), olayout, old, G, m_max, n, k, stream)
    _check(st, "gemm_grouped_masked_silu_mul_quant")
    return out, out_scale


def gemm_grouped_contiguous_mxfp4_raw(a_ptr, sa_ptr, b_ptr, sb_ptr, layout_ptr, d_ptr, out_dtype,
                                      m_sum, n, k, num_groups, stream=None) -> int:
    lib = load()
    return lib.gemm_grouped_contiguous_mxfp4(a_ptr, sa_ptr, b_ptr, sb_ptr, layout_ptr, d_ptr,
                                             int(out_dtype), int(m_sum), int(n), int(k),
                                             int(num_groups), ctypes.c_void_p(_stream_handle(stream)))


def gemm_grouped_masked_mxfp4_raw(a_ptr, sa_ptr, b_ptr, sb_ptr, masked_m_ptr, expected_m, d_ptr,
                                  out_dtype, num_groups, m_max, n, k, stream=None) -> int:
    lib = load()
    return lib.gemm_grouped_masked_mxfp4(a_ptr, sa_ptr, b_ptr, sb_ptr, masked_m_ptr,
                                         int(expected_m), d_ptr, int(out_dtype), int(num_groups),
                                         int(m_max), int(n), int(k),
                                         ctypes.c_void_p(_stream_handle(stream)))


def _u8(t, name):
    if t.dtype != torch.uint8 or not t.is_contiguous() or not t.is_cuda:
        raise TypeError(f"{name} must be a contiguous uint8 CUDA tensor")
    return t.data_ptr()


def gemm_grouped_contiguous_mxfp4(a, scale_a, b, scale_b, d, grouped_layout, *, stream=None):
    """MXFP4 grouped GEMM, contiguous variant (include/fp8bs.h).

    a uint8 [M_sum, K/2] packed E2M1 (element 2i in the low nibble); scale_a uint8
    [M_sum, K/32] E8M0; b uint8 [G, N, K/2]; scale_b uint8 [G, N, K/32]; d bf16/f16
    [M_sum, N]; grouped_layout int32 [M_sum], -1 = padding (not written).
    """
    m_sum, kh = a.shape
    G, n, kh2 = b.shape
    k = 2 * kh
    if kh2 != kh or scale_a.shape != (m_sum, k // 32) or scale_b.shape != (G, n, k // 32):
        raise ValueError("shape mismatch")
    if d.shape != (m_sum, n) or not d.is_contiguous() or grouped_layout.shape != (m_sum,):
        raise ValueError("d must be contiguous [M_sum, N], grouped_layout [M_sum]")
    if grouped_layout.dtype != torch.int32:
        raise ValueError("grouped_layout must be int32")
    dev = _device_of(a, scale_a, b, scale_b, d, grouped_layout, stream=stream)
    with torch.cuda.device(dev):
        st = gemm_grouped_contiguous_mxfp4_raw(_u8(a, "a"), _u8(scale_a, "scale_a"), _u8(b, "b"),
                                               _u8(scale_b, "scale_b"),
                                               _contig_ptr(grouped_layout, "grouped_layout"),
                                               d.data_ptr(), _out_code(d), m_sum, n, k, G, stream)
    _check(st, "gemm_grouped_contiguous_mxfp4")
    return d


def gemm_grouped_masked_mxfp4(a, scale_a, b, scale_b, d, masked_m, expected_m: int = 0, *,
                              stream=None):
    """MXFP4 grouped GEMM, masked variant: a [G, M_max, K/2], scale_a [G, M_max, K/32],
    d [G, M_max, N]; rows m >= masked_m[g] are not written."""
    G, m_max, kh = a.shape
    Gb, n, kh2 = b.shape
    k = 2 * kh
    if Gb != G or kh2 != kh or scale_a.shape != (G, m_max, k // 32) or scale_b.shape != (G, n, k // 32):
        raise ValueError("shape mismatch")
    if d.shape != (G, m_max, n) or not d.is_contiguous() or masked_m.shape != (G,):
        raise ValueError("d must be contiguous [G, M_max, N], masked_m [G]")
    if masked_m.dtype != torch.int32:
        raise ValueError("masked_m must be int32")
    dev = _device_of(a, scale_a, b, scale_b, d, masked_m, stream=stream)
    with torch.cuda.device(dev):
        st = gemm_grouped_masked_mxfp4_raw(_u8(a, "a"), _u8(scale_a, "scale_a"), _u8(b, "b"),
                                           _u8(scale_b, "scale_b"),
                                           _contig_ptr(masked_m, "masked_m"), expected_m,
                                           d.data_ptr(), _out_code(d), G, m_max, n, k, stream)
    _check(st, "gemm_grouped_masked_mxfp4")
    return d


def device_error(device: int = None) -> int:
    """Synchronise the device and return (and clear) its FP8BS_DEVERR_* bits."""
    lib = load()
    if device is None:
        device = torch.cuda.current_device()
    flags = ctypes.c_uint32(0)
    st = lib.fp8bs_device_error(int(device), ctypes.byref(flags))
    if st not in (0, 4):
        raise Fp8bsError(st, "fp8bs_device_error")
    return int(flags.value)


DEBUG_STALL_MMA = 0x1
DEBUG_SINGLE_CTA = 0x2


def set_debug_flags(flags: int) -> None:
    """Test hook (include/fp8bs.h): DEBUG_STALL_MMA makes later pair-kernel launches
    time out and abort on purpose; DEBUG_SINGLE_CTA routes the plain entry points to
    the single-CTA kernel; 0 turns both off."""
    _check(load().fp8bs_set_debug_flags(int(flags)), "fp8bs_set_debug_flags")


def clear_cache() -> None:
    _check(load().fp8bs_clear_cache(), "fp8bs_clear_cache")


def abi_version() -> int:
    return int(load().fp8bs_abi_version())


def kernel_launches() -> int:
    """Kernels the library has launched in this process (a host-side counter)."""
    return int(load().fp8bs_kernel_launches())
