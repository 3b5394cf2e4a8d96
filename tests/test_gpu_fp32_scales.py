"""GPU parity of the software-promotion kernel (arbitrary fp32 block scales),
called through the C ABI, against the CPU oracle, with the tolerances of the
other parity tests (_parity.py); and a cross-check of the hardware-scaled
kernel against it on power-of-two scales."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_gb300 as fb
import oracle
import synth
from synth.inputs import SA_KM, SA_MK

from _parity import all_rows, compare, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM], ids=["sa_mk", "sa_km"])
@pytest.mark.parametrize("out", [0, 1], ids=["bf16", "f16"])
def test_contiguous_fp32_scales_ragged(gg, sa_layout, out):
    # K = 384: three K blocks, so a stage holds a lone last block
    p = synth.make_problem("contiguous", 3, 512, 384, [100, 300, 257], out_dtype=out,
                           sa_layout=sa_layout, seed=401, device=DEV, tail_rows=30,
                           scale_kind="fp32")
    assert np.any(np.frexp(p.sb.cpu().numpy())[0] != 0.5)
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    print(compare(p, bits, valid, untouched))


def test_contiguous_fp32_scales_many_rounds(gg):
    # 10 pair tiles x 8 column tiles = 80 units: more than one round on 76 pairs, so the
    # two partial buffers alternate across units
    p = synth.make_problem("contiguous", 2, 2048, 1024, [1280, 1200], sa_layout=SA_KM, seed=402,
                           device=DEV, scale_kind="fp32")
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    print(compare(p, bits, valid, untouched))
    assert np.array_equal(bits, run_gpu(p))   # deterministic


@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM], ids=["sa_mk", "sa_km"])
def test_masked_fp32_scales(gg, sa_layout):
    p = synth.make_problem("masked", 4, 768, 512, [0, 1, 150, 300], sa_layout=sa_layout,
                           seed=403, M_max=300, device=DEV, scale_kind="fp32")
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    print(compare(p, bits, valid, untouched))


def test_promotion_agrees_with_hardware_scaling(gg):
    """On power-of-two scales both kernels compute the same values; each is checked
    against the oracle, and the two must agree element-wise within the same bound."""
    p = synth.make_problem("contiguous", 2, 1024, 1024, [256, 300], seed=404, device=DEV)
    hw = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, hw, valid, untouched)
    d = torch.full((p.rows, p.N), 0x7FA5, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    fb.gemm_grouped_contiguous_fp32_scales(p.a, p.sa_mk_view(), p.b, p.sb, d, p.grouped_layout)
    torch.cuda.synchronize()
    assert fb.device_error() == 0
    sw = d.view(torch.int16).cpu().numpy().view(np.uint16)
    compare(p, sw, valid, untouched)
    x = oracle.bits_to_float(hw[valid], 0)
    y = oracle.bits_to_float(sw[valid], 0)
    assert oracle.calc_diff(x, y) <= 1e-5
    # bf16 results of two fp32 accumulation orders: mostly identical, never far apart
    assert np.mean(hw[valid] == sw[valid]) >= 0.9
    assert np.all(np.abs(x - y) <= 2.0 ** -7 * np.abs(x) + 1e-2 * np.sqrt(np.mean(x * x)))


def test_fp32_scales_empty(gg):
    p = synth.make_problem("contiguous", 1, 256, 256, [128], seed=405, device=DEV,
                           scale_kind="fp32")
    d = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    fb.gemm_grouped_contiguous_fp32_scales(p.a[:0], p.sa_mk_view()[:0], p.b, p.sb, d,
                                           p.grouped_layout[:0])
    torch.cuda.synchronize()
