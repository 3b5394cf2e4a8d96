"""gemm_grouped_contiguous_noalloc: the entry point for callers that may not
allocate device memory (it keeps its scratch in a static device array of the
library).  Through the C ABI, two calls in a row must match the allocating
entry point gemm_grouped_contiguous within the parity tolerances of the other
GPU tests, and each call's valid rows must also meet those tolerances against
the CPU oracle directly (a fault that both entry points shared would otherwise
go unseen).  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_gb300 as fb
import oracle
import synth
from fp8_block_scaled_gb300 import _binding
from synth.inputs import OUT_F16, SA_KM, SA_MK

from _parity import CALC_DIFF_ORACLE, REL_TOL, RMS_TOL, SENTINEL, all_rows, compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(raw_fn, p, d_offset=0):
    numel = p.rows * p.N
    full = torch.full((numel + 16,), SENTINEL, dtype=torch.int16, device=DEV)
    buf = full[d_offset:d_offset + numel]
    d = buf.view(torch.bfloat16 if p.out_dtype == 0 else torch.float16)
    layout, ld = _binding._sa_layout_2d(p.sa_mk_view(), p.rows, p.KB)
    st = raw_fn(p.a.data_ptr(), p.sa.data_ptr(), layout, ld, p.b.data_ptr(), p.sb.data_ptr(),
                p.grouped_layout.data_ptr(), d.data_ptr(), p.out_dtype, p.rows, p.N, p.K, p.G)
    assert st == 0, fb.status_string(st)
    torch.cuda.synchronize()
    assert fb.device_error() == 0
    around = torch.cat([full[:d_offset], full[d_offset + numel:]]).cpu().numpy().view(np.uint16)
    assert (around == SENTINEL).all(), "a word outside D was written"
    return buf.cpu().numpy().view(np.uint16).reshape(p.rows, p.N)


PROBLEMS = [
    # 80 units of 256 x 256: the stream-K split (and so the scratch) is used on 76 CTA pairs
    dict(G=2, N=2560, K=1024, sizes=[1024, 1000], sa_layout=SA_KM, out=0, seed=201),
    # ragged experts, f16 output, row-major activation scales
    dict(G=3, N=512, K=768, sizes=[100, 300, 257], sa_layout=SA_MK, out=OUT_F16, seed=202),
    # N % 256 == 128: a 128-column last tile
    dict(G=2, N=384, K=512, sizes=[300, 129], sa_layout=SA_KM, out=0, seed=203),
    # D only 16-byte aligned (8 elements into its buffer): 16-byte stores
    dict(G=2, N=512, K=512, sizes=[256, 200], sa_layout=SA_KM, out=0, seed=204, d_offset=8),
]


@pytest.mark.parametrize("spec", PROBLEMS, ids=["streamk_80_units", "ragged_f16", "n384", "d16"])
def test_noalloc_matches_allocating_entry_point_twice(gg, spec):
    p = synth.make_problem("contiguous", spec["G"], spec["N"], spec["K"], spec["sizes"],
                           out_dtype=spec["out"], sa_layout=spec["sa_layout"], seed=spec["seed"],
                           device=DEV)
    off = spec.get("d_offset", 0)
    ref_bits = _run(_binding.gemm_grouped_contiguous_raw, p, off)
    valid, untouched = all_rows(p)
    ref = oracle.bits_to_float(ref_bits[valid], p.out_dtype)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    for _ in range(2):
        bits = _run(_binding.gemm_grouped_contiguous_noalloc_raw, p, off)
        got = oracle.bits_to_float(bits[valid], p.out_dtype)
        assert np.isfinite(got).all()
        assert oracle.calc_diff(got, ref) <= CALC_DIFF_ORACLE
        assert (np.abs(got - ref) <= REL_TOL * np.abs(ref) + RMS_TOL * rms).all()
        assert (bits[untouched] == SENTINEL).all()
        compare(p, bits, valid, untouched, check_fp32=False)  # against the oracle itself
