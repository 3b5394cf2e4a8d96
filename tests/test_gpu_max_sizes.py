"""GPU parity at the contiguous pair kernels' list limits and past them.

The CTA-pair kernels keep their list of expert tile pairs in shared memory for
up to 4096 row tiles of 128 (3968 for MXFP4), and in a per-stream device
workspace above that (up to 32768 tiles).  Problems at the shared-memory limit,
one tile past it and far past it are checked against the oracle on seeded
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


def test_pair_list_in_workspace_one_tile_past_the_limit(gg):
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


def test_workspace_list_a_million_rows(gg):
    # 8192 row tiles: the pair list in the workspace, grouped_layout read in two rounds
    p = synth.make_problem("contiguous", 128, 256, 256, [8192] * 128, seed=616, device=DEV)
    assert p.rows == 2 * PAIR_MAX_ROWS
    print(_check(p, 5))


@pytest.mark.parametrize("kind", ["mxfp4", "fp32"])
def test_variant_paths_past_the_shared_memory_list(gg, kind):
    sizes = [8192] * 63 + [8193] if kind == "fp32" else [8192] * 62 + [1]
    p = synth.make_problem("contiguous", len(sizes), 256, 256, sizes, seed=617, device=DEV,
                           scale_kind=kind)
    assert p.rows == (PAIR_MAX_ROWS if kind == "fp32" else 3968 * 128) + 128
    print(_check(p, 6))
