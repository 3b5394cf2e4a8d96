"""GPU parity at the contiguous pair path's size limit and just past it.

The CTA-pair kernel keeps its list of expert tile pairs in shared memory, at
most 4096 tiles of 128 rows (m_sum <= 524288).  A problem of exactly that many
tiles must run on it; one tile more must fall back to the single-CTA kernel,
which has no such list.  Both are checked against the oracle on seeded
samples of rows (group edges + random rows) and on the untouched padding rows.
"""
import pytest

import synth

from _parity import compare, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"
PAIR_MAX_ROWS = 4096 * 128


def _check(p, seed):
    """Sampled rows include every expert's first and last valid row and its first
    and last padding row (the ragged tail of the last tile among them)."""
    bits = run_gpu(p)
    valid, untouched = synth.sample_rows(p, per_group=8, seed=seed)
    return compare(p, bits, valid, untouched)


def test_pair_path_at_the_tile_limit(gg):
    # 64 experts x 8192 rows: exactly 4096 row tiles
    p = synth.make_problem("contiguous", 64, 256, 256, [8192] * 64, seed=611, device=DEV)
    assert p.rows == PAIR_MAX_ROWS
    print(_check(p, 1))


def test_single_cta_fallback_one_tile_past_the_limit(gg):
    # one expert one row longer: 4097 row tiles, the last expert ragged
    sizes = [8192] * 63 + [8193]
    p = synth.make_problem("contiguous", 64, 256, 256, sizes, seed=612, device=DEV)
    assert p.rows == PAIR_MAX_ROWS + 128
    print(_check(p, 2))


def test_mxfp4_at_its_tile_limit(gg):
    # the MXFP4 pair list holds 3968 row tiles (larger scale staging): 62 x 8192 rows
    p = synth.make_problem("contiguous", 62, 256, 256, [8192] * 62, seed=613, device=DEV,
                           scale_kind="mxfp4")
    assert p.rows == 3968 * 128
    print(_check(p, 3))


def test_fp32_scales_at_the_tile_limit(gg):
    # the promotion kernel shares the pair list (4096 row tiles)
    p = synth.make_problem("contiguous", 64, 256, 256, [8192] * 64, seed=614, device=DEV,
                           scale_kind="fp32")
    assert p.rows == PAIR_MAX_ROWS
    print(_check(p, 4))
