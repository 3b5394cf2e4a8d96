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


def _embed_groups(p, G, ids):
    """p's experts as experts `ids` of a G-expert problem: the other experts' weights
    are zero with unit scales and own no rows, so every row's result is p's."""
    import torch
    b = torch.zeros((G,) + tuple(p.b.shape[1:]), dtype=p.b.dtype, device=DEV)
    sb = torch.ones((G,) + tuple(p.sb.shape[1:]), dtype=torch.float32, device=DEV)
    idx = torch.tensor(ids, device=DEV)
    b[idx] = p.b
    sb[idx] = p.sb
    return b, sb, idx


@pytest.mark.parametrize("G", [(1 << 15) - 1, 1 << 15])
def test_contiguous_expert_ids_at_the_pair_list_limit(gg, G):
    """A pair-list entry holds the expert id in 15 bits: 32767 experts run on the
    CTA-pair kernel (ids up to 32766 in use), 32768 on the single-CTA kernel."""
    import numpy as np
    import torch
    import fp8_block_scaled_gb300 as fb
    from _parity import SENTINEL, all_rows
    p = synth.make_problem("contiguous", 3, 256, 256, [100, 130, 60], seed=618, device=DEV,
                           tail_rows=20)
    ids = [0, G // 2, G - 1]
    b, sb, idx = _embed_groups(p, G, ids)
    layout = torch.where(p.grouped_layout >= 0, idx[p.grouped_layout.clamp(min=0).long()],
                         p.grouped_layout).to(torch.int32)
    d = torch.full((p.rows, p.N), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    fb.gemm_grouped_contiguous(p.a, p.sa_mk_view(), b, sb, d, layout)
    torch.cuda.synchronize()
    assert fb.device_error() == 0
    bits = d.view(torch.int16).cpu().numpy().view(np.uint16)
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched)


def test_masked_at_its_group_limit(gg):
    """1024 groups (the masked kernels' limit), rows in a few of them."""
    import numpy as np
    import torch
    import fp8_block_scaled_gb300 as fb
    from _parity import SENTINEL
    G, ids = 1024, [0, 511, 1023]
    p = synth.make_problem("masked", 3, 256, 256, [70, 200, 1], M_max=200, seed=619, device=DEV)
    b, sb, idx = _embed_groups(p, G, ids)
    a = torch.zeros((G, p.M_max, p.K), dtype=p.a.dtype, device=DEV)
    a[idx] = p.a
    sa = torch.ones((G, p.M_max, p.KB), dtype=torch.float32, device=DEV)
    sa[idx] = p.sa_mk_view()
    mm = torch.zeros(G, dtype=torch.int32, device=DEV)
    mm[idx] = p.masked_m
    d = torch.full((G, p.M_max, p.N), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    fb.gemm_grouped_masked(a, sa, b, sb, d, mm)
    torch.cuda.synchronize()
    assert fb.device_error() == 0
    out = d.view(torch.int16).cpu().numpy().view(np.uint16)
    # the three groups in use, against the oracle; every other group untouched
    bits = out[ids].reshape(-1, p.N)
    from _parity import all_rows
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched)
    rest = np.setdiff1d(np.arange(G), ids)
    assert (out[rest] == SENTINEL).all()
