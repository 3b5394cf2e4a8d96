"""Failure detection without a GPU fault: the test hook FP8BS_DEBUG_STALL_MMA
makes the CTA-pair kernel's MMA thread wait on a barrier nothing arrives on.
The wait gives up after its time limit, the launch aborts cleanly (every other
wait sees the abort flag, copies land, tensor memory is freed), the host reads
FP8BS_DEVERR_TIMEOUT, and the context stays usable: the next launch is correct."""
import time

import numpy as np
import pytest
import torch

import fp8_block_scaled_gb300 as fb
import synth

from _parity import all_rows, compare, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_stalled_wait_times_out_and_the_context_survives(gg):
    # 80 units on 76 pairs: the stream-K split is armed when the abort happens
    p = synth.make_problem("contiguous", 2, 2560, 512, [1024, 1000], seed=601, device=DEV)
    fb.device_error()            # start from a clear error word
    fb.set_debug_flags(fb.DEBUG_STALL_MMA)
    try:
        d = torch.zeros((p.rows, p.N), dtype=torch.bfloat16, device=DEV)
        t0 = time.time()
        fb.gemm_grouped_contiguous(p.a, p.sa_mk_view(), p.b, p.sb, d, p.grouped_layout)
        torch.cuda.synchronize()
        waited = time.time() - t0
    finally:
        fb.set_debug_flags(0)
    assert fb.device_error() & fb.DEVERR_TIMEOUT
    assert 3.0 < waited < 60.0, waited
    # the same problem again, through the same library state
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched)


def test_debug_flags_reject_unknown_bits(gg):
    with pytest.raises(fb.Fp8bsError):
        fb.set_debug_flags(0x80)
