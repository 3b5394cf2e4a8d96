"""GPU parity of the MXFP4 (a4w4) grouped GEMM -- packed E2M1 operands with E8M0
scales per 32 elements, tcgen05.mma kind::mxf4 -- called through the C ABI,
against the CPU oracle (tolerances of _parity.py; the pre-quantisation check
uses the MXFP4 bound there)."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_gb300 as fb
import synth

from _parity import all_rows, compare, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(p):
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    stats = compare(p, bits, valid, untouched)
    print(stats)
    return bits


def test_one_k_block(gg):
    # K = 256: a single K block (four kind::mxf4 MMAs, both scale words)
    _check(synth.make_problem("contiguous", 2, 256, 256, [100, 200], seed=501, device=DEV,
                              scale_kind="mxfp4"))


@pytest.mark.parametrize("out", [0, 1], ids=["bf16", "f16"])
def test_ragged_three_k_blocks(gg, out):
    # K = 768: three K blocks, so the last stage holds one; ragged groups and tail rows
    _check(synth.make_problem("contiguous", 3, 512, 768, [100, 300, 257], out_dtype=out,
                              seed=502, device=DEV, tail_rows=40, scale_kind="mxfp4"))


def test_long_k(gg):
    _check(synth.make_problem("contiguous", 2, 512, 7168, [256, 130], seed=503, device=DEV,
                              scale_kind="mxfp4"))


def test_stream_k_split(gg):
    # 16 pair tiles x 10 column tiles = 160 units on 76 pairs: the stream-K tail runs
    p = synth.make_problem("contiguous", 2, 2560, 1024, [1024, 1000], seed=504, device=DEV,
                           scale_kind="mxfp4")
    bits = _check(p)
    assert np.array_equal(bits, run_gpu(p))


def test_masked(gg):
    _check(synth.make_problem("masked", 4, 512, 512, [0, 1, 150, 300], seed=505, M_max=300,
                              device=DEV, scale_kind="mxfp4"))


def test_masked_equals_contiguous_bitwise(gg):
    pc = synth.make_problem("contiguous", 2, 512, 512, [256, 256], seed=506, device=DEV,
                            scale_kind="mxfp4")
    pm = synth.make_problem("masked", 2, 512, 512, [256, 256], seed=506, M_max=256, device=DEV,
                            scale_kind="mxfp4")
    assert np.array_equal(run_gpu(pc), run_gpu(pm))


def test_empty(gg):
    p = synth.make_problem("contiguous", 1, 256, 256, [128], seed=507, device=DEV,
                           scale_kind="mxfp4")
    d = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    fb.gemm_grouped_contiguous_mxfp4(p.a[:0], p.sa[:0], p.b, p.sb, d, p.grouped_layout[:0])
    torch.cuda.synchronize()
