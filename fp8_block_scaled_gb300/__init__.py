"""GB300-native (sm_103a) grouped FP8 block-scaled GEMM for MoE expert projections.

The operation is the one of "Adds Grouped and Batched GEMM kernels with
blockscaling matching DeepGEMM API" (FlyDSL PR #433), section Summary:

    D[r, n] = sum_kb scale_a[r, kb] * scale_b[g, n/128, kb]
                     * sum_{k in block kb} A[r, k] * B[g, n, k]

E4M3 operands, (1,128) activation and (128,128) weight UE8M0 scales, fp32
accumulation, bf16/f16 output, in a contiguous (grouped_layout, -1 = padding)
and a masked (masked_m) variant.  All compute runs in the hand-written CUDA
kernels of ``libfp8bs.so``; this package only marshals arguments.  The
``*_silu_mul_quant`` entry points fuse the first MoE GEMM's SiLU(gate) * up and
the (1,128) E4M3 requantisation of its output into the same kernel; the
``*_fp32_scales`` entry points take arbitrary fp32 block scales (promoted in
software instead of by the tensor core); the ``*_mxfp4`` entry points take both
operands in MXFP4 (E2M1 with E8M0 scales per 32 elements).
"""
from ._binding import (  # noqa: F401
    DEBUG_SINGLE_CTA,
    DEBUG_STALL_MMA,
    DEVERR_BAD_GROUP,
    DEVERR_BAD_SCALE,
    DEVERR_MASKED_M,
    DEVERR_MIXED_TILE,
    DEVERR_TIMEOUT,
    EXPORTS,
    OUT_BF16,
    OUT_F16,
    SA_KM,
    SA_MK,
    Fp8bsError,
    abi_version,
    clear_cache,
    device_error,
    gemm_grouped_contiguous,
    gemm_grouped_contiguous_fp32_scales,
    gemm_grouped_contiguous_fp32_scales_raw,
    gemm_grouped_contiguous_mxfp4,
    gemm_grouped_contiguous_mxfp4_raw,
    gemm_grouped_contiguous_noalloc_raw,
    gemm_grouped_contiguous_raw,
    gemm_grouped_contiguous_silu_mul_quant,
    gemm_grouped_contiguous_silu_mul_quant_raw,
    gemm_grouped_masked,
    gemm_grouped_masked_fp32_scales,
    gemm_grouped_masked_fp32_scales_raw,
    gemm_grouped_masked_mxfp4,
    gemm_grouped_masked_mxfp4_raw,
    gemm_grouped_masked_raw,
    gemm_grouped_masked_silu_mul_quant,
    gemm_grouped_masked_silu_mul_quant_raw,
    kernel_launches,
    lib_path,
    load,
    set_debug_flags,
    status_string,
)
