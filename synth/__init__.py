"""Seeded synthetic inputs for the grouped FP8 block-scaled GEMM.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__``.  It
holds the input recipe only -- random draws, the group-size draws and the
host-side quantisation of fp32 data into e4m3 codes with UE8M0 scales -- and
none of the GEMM's arithmetic.  Neither the oracle nor the CUDA library
imports it; both consume the tensors it returns.

Recipe ("Adds Grouped and Batched GEMM kernels with blockscaling matching
DeepGEMM API", FlyDSL PR #433, *DeepGEMM conformance details*): fp32 data
~ N(0, 1); per (1, 128) block of A and per (128, 128) block of B,
``amax = max|x|`` (clamped below at 1e-4), ``s = ceil_to_ue8m0(amax / 448)``,
``q = e4m3(x / s)`` with round-to-nearest-even.  The ceiling keeps
``|x / s| <= 448`` so nothing saturates.
"""
from .inputs import (  # noqa: F401
    CONFIGS,
    Problem,
    ceil_to_ue8m0_f32,
    draw_group_sizes,
    make_config,
    make_problem,
    quantize_a_blocks,
    quantize_b_blocks,
    sample_rows,
)
