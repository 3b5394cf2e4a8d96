"""GPU parity: the sm_103a kernels, called through the C ABI, against the CPU
oracle on the same seeded inputs (see _parity.py for the tolerances).

Small problems are compared on every row; the named workloads at full
size are compared on seeded samples of rows (group edges + random rows), in
the same launch configuration bench.py times.
"""
import json
import os

import numpy as np
import pytest
import torch

import fp8_block_scaled_gb300 as fb
import oracle
import synth
from synth.inputs import OUT_BF16, OUT_F16, SA_KM, SA_MK

from _parity import SENTINEL, all_rows, compare, run_gpu, single_cta_kernel

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_config1_all_rows(gg):
    p = synth.make_config("c1_contig_g2_m100_n256_k256", device=DEV)
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    stats = compare(p, bits, valid, untouched)
    assert valid.size == 200 and untouched.size == 56
    assert stats["exact_frac"] > 0.9


@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM])
@pytest.mark.parametrize("out", [OUT_BF16, OUT_F16])
def test_contiguous_ragged_multi_tile(gg, sa_layout, out):
    """Several m/n tiles, an empty expert, an expert spanning 3 tiles, a ragged
    M_sum tail of -1 rows, N=384 (a 128-column last tile on the CTA-pair kernel)."""
    p = synth.make_problem("contiguous", 3, 384, 512, [130, 0, 300], out_dtype=out,
                           sa_layout=sa_layout, seed=31 + out, tail_rows=37, device=DEV)
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched)


@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM])
def test_contiguous_wide_n_tiles(gg, sa_layout):
    """N=768 (256-column tiles), K=1024, 4 experts of unaligned sizes."""
    p = synth.make_problem("contiguous", 4, 768, 1024, [1, 127, 129, 256], sa_layout=sa_layout,
                           seed=41, device=DEV)
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched)


@pytest.mark.parametrize("out", [OUT_BF16, OUT_F16])
@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM])
@pytest.mark.parametrize("n", [256, 384])
def test_masked_ragged(gg, sa_layout, n, out):
    """M_max=200 (not a multiple of 128); masked_m = 0, 1, 200 (full) and 129."""
    p = synth.make_problem("masked", 4, n, 384, [0, 1, 200, 129], M_max=200, out_dtype=out,
                           sa_layout=sa_layout, seed=51, device=DEV)
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched)


@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM])
def test_masked_m_at_half_tile_edges(gg, sa_layout):
    """masked_m just below, at and above multiples of 128: the pairs whose second
    128 rows hold no computed row (masked_m % 256 in [1, 128]) load no A there."""
    sizes = [128, 129, 256, 257, 384, 385, 511, 512]
    p = synth.make_problem("masked", len(sizes), 512, 512, sizes, M_max=512, sa_layout=sa_layout,
                           seed=57, device=DEV)
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched)


def test_masked_full_equals_contiguous_bitwise(gg):
    G, M, N, K = 3, 256, 512, 512
    pc = synth.make_problem("contiguous", G, N, K, [M] * G, seed=61, device=DEV)
    pm = synth.make_problem("masked", G, N, K, [M] * G, M_max=M, seed=61, device=DEV)
    assert torch.equal(pc.a.reshape(G, M, K), pm.a) and torch.equal(pc.b, pm.b)
    bc = run_gpu(pc)
    bm = run_gpu(pm)
    assert np.array_equal(bc, bm)


def test_deterministic(gg):
    p = synth.make_problem("contiguous", 2, 512, 768, [200, 300], seed=71, device=DEV)
    assert np.array_equal(run_gpu(p), run_gpu(p))


def test_empty_inputs_are_noops(gg):
    p = synth.make_problem("masked", 3, 256, 256, [0, 0, 0], M_max=64, seed=81, device=DEV)
    bits = run_gpu(p)
    assert (bits == SENTINEL).all()
    a = torch.empty((0, 256), dtype=torch.uint8, device=DEV)
    sa = torch.empty((0, 2), dtype=torch.float32, device=DEV)
    d = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    lay = torch.empty((0,), dtype=torch.int32, device=DEV)
    q = synth.make_problem("contiguous", 1, 256, 256, [1], seed=82, device=DEV)
    fb.gemm_grouped_contiguous(a, sa, q.b, q.sb, d, lay)
    torch.cuda.synchronize()
    assert fb.device_error() == 0


def _fill(spec, shape):
    arr = np.empty(shape, dtype=np.uint8)
    arr[...] = spec["default"]
    for ranges, code in spec.get("fill", []):
        arr[tuple(slice(lo, hi) for lo, hi in ranges)] = code
    return arr


with open(os.path.join(GOLDEN, "hand_cases.json")) as _f:
    _HAND = json.load(_f)["cases"]


@pytest.mark.parametrize("case", [c for c in _HAND if c.get("tile_aligned", True)],
                         ids=lambda c: c["name"])
def test_hand_cases_exact_bits(gg, case):
    """The hand-derived golden cases: the kernel's output bits equal the
    expected bits exactly (all of them are exact in fp32 accumulation)."""
    K, N, G = case["K"], case["N"], case["G"]
    b = torch.from_numpy(_fill(case["b_codes"], (G, N, K))).to(DEV)
    sb = torch.tensor(case["scale_b"], dtype=torch.float32, device=DEV).reshape(G, N // 128, K // 128)
    dt = torch.bfloat16 if case["out_dtype"] == 0 else torch.float16
    if case["variant"] == "contiguous":
        M = len(case["grouped_layout"])
        a = torch.from_numpy(_fill(case["a_codes"], (M, K))).to(DEV)
        sa = torch.tensor(case["scale_a"], dtype=torch.float32, device=DEV).reshape(M, K // 128)
        lay = torch.tensor(case["grouped_layout"], dtype=torch.int32, device=DEV)
        d = torch.full((M, N), SENTINEL, dtype=torch.int16, device=DEV).view(dt)
        fb.gemm_grouped_contiguous(a, sa, b, sb, d, lay)
    else:
        Mx = case["M_max"]
        a = torch.from_numpy(_fill(case["a_codes"], (G, Mx, K))).to(DEV)
        sa = torch.tensor(case["scale_a"], dtype=torch.float32, device=DEV).reshape(G, Mx, K // 128)
        mm = torch.tensor(case["masked_m"], dtype=torch.int32, device=DEV)
        d = torch.full((G, Mx, N), SENTINEL, dtype=torch.int16, device=DEV).view(dt)
        fb.gemm_grouped_masked(a, sa, b, sb, d, mm)
    torch.cuda.synchronize()
    assert fb.device_error() == 0
    bits = d.view(torch.int16).reshape(-1, N).cpu().numpy().view(np.uint16)
    for r, ok in enumerate(case["valid"]):
        if not ok:
            assert (bits[r] == SENTINEL).all()
    for r, expect in case["expect_rows"].items():
        for lo, hi, value, hexbits in expect["segments"]:
            assert (bits[int(r), lo:hi] == int(hexbits, 16)).all(), (r, hex(int(bits[int(r), lo])))


# (D offset in elements, single-CTA kernel): a 32-byte aligned D on the CTA-pair
# kernel, a 16-byte aligned D on the CTA-pair kernel (its 16-byte stores), and the
# single-CTA kernel (test hook)
KERNELS = [pytest.param(0, False, id="pair"), pytest.param(8, False, id="pair_d16"),
           pytest.param(0, True, id="single_cta")]


@pytest.mark.parametrize("d_offset,single", KERNELS)
def test_device_flags_mixed_and_bad_groups(gg, d_offset, single):
    """The first row of a 128-row tile names its expert (the contiguous layout
    pads every expert to a multiple of 128 rows).  A row of another expert
    inside a tile, and a group id out of range, are reported in the device
    error word and left unwritten, by both kernels and with either D alignment."""
    p = synth.make_problem("contiguous", 2, 256, 256, [128, 128], seed=91, device=DEV)
    lay = p.grouped_layout.clone()
    lay[5] = 1            # tile 0 (expert 0) now holds a row of expert 1
    lay[200] = 7          # out of range in tile 1 (expert 1)
    buf = torch.full((256 * 256 + 16,), SENTINEL, dtype=torch.int16, device=DEV)
    d = buf[d_offset:d_offset + 256 * 256].view(torch.bfloat16).view(256, 256)
    with single_cta_kernel(single):
        fb.gemm_grouped_contiguous(p.a, p.sa, p.b, p.sb, d, lay)
    torch.cuda.synchronize()
    flags = fb.device_error()
    assert flags & fb.DEVERR_MIXED_TILE and flags & fb.DEVERR_BAD_GROUP
    bits = d.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (bits[5] == SENTINEL).all() and (bits[200] == SENTINEL).all()
    assert (bits[:5] != SENTINEL).all() and (bits[6:200] != SENTINEL).all()
    assert (bits[201:] != SENTINEL).all()
    assert fb.device_error() == 0  # cleared by the read


@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM])
@pytest.mark.parametrize("n", [512, 384])
@pytest.mark.parametrize("variant", ["contiguous", "masked"])
def test_single_cta_and_pair_kernels_agree(gg, variant, n, sa_layout):
    """The same problem through the CTA-pair kernel with a 32-byte and a 16-byte
    aligned D (one 32-byte store or two 16-byte stores per 16 columns) and through
    the single-CTA kernel, each against the oracle; the two pair runs are
    bit-identical and the words around D are never written.  With row-major
    activation scales the pair kernel reads the scale pre-pass's images, the
    single-CTA kernel converts the scales itself."""
    if variant == "contiguous":
        p = synth.make_problem("contiguous", 3, n, 768, [100, 300, 257], sa_layout=sa_layout,
                               seed=93, device=DEV)
        shape = (p.rows, p.N)
    else:
        p = synth.make_problem("masked", 3, n, 768, [100, 300, 257], M_max=320,
                               sa_layout=sa_layout, seed=94, device=DEV)
        shape = (p.G, p.M_max, p.N)
    numel = p.rows * p.N
    outs = []
    for off, single in ((0, False), (8, False), (0, True)):
        buf = torch.full((numel + 32,), SENTINEL, dtype=torch.int16, device=DEV)
        d = buf[off:off + numel].view(torch.bfloat16).view(*shape)
        with single_cta_kernel(single):
            if variant == "contiguous":
                fb.gemm_grouped_contiguous(p.a, p.sa_mk_view(), p.b, p.sb, d, p.grouped_layout)
            else:
                fb.gemm_grouped_masked(p.a, p.sa_mk_view(), p.b, p.sb, d, p.masked_m)
        torch.cuda.synchronize()
        assert fb.device_error() == 0
        whole = buf.cpu().numpy().view(np.uint16)
        assert (whole[:off] == SENTINEL).all() and (whole[off + numel:] == SENTINEL).all()
        outs.append(whole[off:off + numel].reshape(-1, p.N))
    valid, untouched = all_rows(p)
    for bits in outs:
        compare(p, bits, valid, untouched, check_fp32=False)
    assert np.array_equal(outs[0], outs[1])
    assert (outs[0] == outs[2]).mean() > 0.99


def test_misaligned_d_at_full_size(gg):
    """The headline workload with D only 16-byte aligned (a slice of a larger
    buffer): the CTA-pair kernel with 16-byte stores, bit-identical to the
    32-byte aligned run, every 128-row tile sampled against the oracle."""
    p = synth.make_config("c2_contig_g8_m1024_n2048_k7168", device=DEV)
    ref = run_gpu(p)
    numel = p.rows * p.N
    buf = torch.full((numel + 16,), SENTINEL, dtype=torch.int16, device=DEV)
    d = buf[8:8 + numel].view(torch.bfloat16).view(p.rows, p.N)
    bits = run_gpu(p, d=d)
    assert np.array_equal(bits, ref)
    assert (buf[:8].cpu().numpy().view(np.uint16) == SENTINEL).all()
    assert (buf[8 + numel:].cpu().numpy().view(np.uint16) == SENTINEL).all()
    valid, untouched = synth.sample_rows(p, per_group=8, seed=3)
    compare(p, bits, valid, untouched, check_fp32=False)


def test_masked_m_out_of_range_is_clamped_and_flagged(gg):
    p = synth.make_problem("masked", 2, 256, 256, [64, 10], M_max=64, seed=92, device=DEV)
    mm = torch.tensor([99, 10], dtype=torch.int32, device=DEV)
    d = torch.full((2, 64, 256), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    fb.gemm_grouped_masked(p.a, p.sa, p.b, p.sb, d, mm)
    torch.cuda.synchronize()
    assert fb.device_error() & fb.DEVERR_MASKED_M
    ref = torch.full_like(d, 0).view(torch.int16).fill_(SENTINEL).view(torch.bfloat16)
    fb.gemm_grouped_masked(p.a, p.sa, p.b, p.sb, ref, p.masked_m)  # masked_m = [64, 10]
    torch.cuda.synchronize()
    assert torch.equal(d.view(torch.int16), ref.view(torch.int16))


# ------------------------------------------------------------------ stream-K tail of the pair kernel
# 80 units of 256 x 256 on a 152-SM GB300 (76 CTA pairs) are not a multiple of
# the pair count, so the units are cut into K runs split across pairs.
def test_stream_k_contiguous_all_rows_and_repeat(gg):
    p = synth.make_problem("contiguous", 2, 2560, 1024, [1024, 1000], sa_layout=SA_KM, seed=101,
                           device=DEV)
    bits1 = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, bits1, valid, untouched, check_fp32=False)
    bits2 = run_gpu(p)  # slot counters were reset by the first launch
    assert np.array_equal(bits1, bits2)


@pytest.mark.parametrize("k", [1024, 1152])
def test_half_column_tile_with_stream_k(gg, k):
    """N = 2432 = 9.5 column tiles of 256: the last tile of every row pair is 128 wide
    (MMA N = 128, each CTA multiplying 64 rows of B), 80 units on 76 CTA pairs, so the
    stream-K split also cuts half-width units; K = 1152 adds an odd count of K blocks."""
    p = synth.make_problem("contiguous", 2, 2432, k, [1024, 1000], sa_layout=SA_KM, seed=104,
                           device=DEV)
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched, check_fp32=False)
    assert np.array_equal(bits, run_gpu(p))


def test_masked_many_units_all_rows(gg):
    """Masked problems always run round-robin (no stream-K split); 80 units."""
    p = synth.make_problem("masked", 4, 2560, 768, [512, 300, 512, 257], M_max=512, seed=102,
                           device=DEV)
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched, check_fp32=False)


def test_stream_k_on_a_second_stream(gg):
    p = synth.make_problem("contiguous", 2, 2560, 1024, [1024, 1000], seed=103, device=DEV)
    ref = run_gpu(p)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        bits = run_gpu(p, stream=side)
    assert np.array_equal(ref, bits)


# ------------------------------------------------------------------ the named workloads, full size
@pytest.mark.parametrize("name", [n for n, c in synth.CONFIGS.items() if not c.get("epilogue")])
def test_named_workload_sampled_rows(gg, name):
    p = synth.make_config(name, device=DEV)
    bits = run_gpu(p)
    if p.rows * p.K <= 4096 * 8192:
        valid, untouched = all_rows(p)
    else:
        valid, untouched = synth.sample_rows(p, per_group=24, seed=1)
    stats = compare(p, bits, valid, untouched)
    print(name, stats)


@pytest.mark.parametrize("sa_layout,kernels", [(SA_MK, 2), (SA_KM, 1)])
def test_kernels_per_call(gg, sa_layout, kernels):
    """Row-major activation scales get the scale pre-pass before the GEMM; the
    transposed layout is read by the GEMM as it is."""
    p = synth.make_problem("contiguous", 2, 512, 512, [200, 150], sa_layout=sa_layout, seed=58,
                           device=DEV)
    run_gpu(p)  # allocates the stream's workspaces
    n0 = fb.kernel_launches()
    bits = run_gpu(p)
    assert fb.kernel_launches() - n0 == kernels
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched)


def test_varying_sizes_on_one_stream(gg):
    """Calls of growing and shrinking sizes on one stream, as a MoE layer sees them
    batch after batch: the stream's workspaces (stream-K scratch, scale images)
    grow and are reused, and every call meets the tolerances on every row."""
    rng = np.random.default_rng(59)
    s = torch.cuda.Stream(priority=-1)
    for i, rows in enumerate([64, 900, 200, 2500, 40, 1300]):
        G = 4
        sizes = [int(v) for v in rng.multinomial(rows, [0.4, 0.3, 0.2, 0.1])]
        K = [512, 1024, 768][i % 3]
        sa_layout = SA_MK if i % 2 == 0 else SA_KM
        p = synth.make_problem("contiguous", G, 512, K, sizes, sa_layout=sa_layout, seed=600 + i,
                               device=DEV)
        with torch.cuda.stream(s):
            bits = run_gpu(p, stream=s)
        valid, untouched = all_rows(p)
        compare(p, bits, valid, untouched, check_fp32=False)


@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM], ids=["sa_mk", "sa_km"])
@pytest.mark.parametrize("n", [128, 384])
@pytest.mark.parametrize("k", [128, 256, 384])
@pytest.mark.parametrize("variant", ["contiguous", "masked"])
def test_smallest_shapes(gg, variant, k, n, sa_layout):
    """The fewest K blocks (one: a pipeline step with an empty second slot; two: one
    step; three: a step and a half) and the narrowest column tiles (N = 128: one
    128-column tile; N = 384: a full tile and a 128-column one), ragged rows."""
    if variant == "contiguous":
        p = synth.make_problem("contiguous", 3, n, k, [1, 130, 77], sa_layout=sa_layout,
                               seed=70 + k // 128 + n, device=DEV, tail_rows=9)
    else:
        p = synth.make_problem("masked", 3, n, k, [1, 130, 0], M_max=140, sa_layout=sa_layout,
                               seed=80 + k // 128 + n, device=DEV)
    bits = run_gpu(p)
    valid, untouched = all_rows(p)
    compare(p, bits, valid, untouched)


def test_expected_m_never_changes_results(gg):
    """expected_m is a hint of the typical masked_m (DeepGEMM's masked contract, as
    "Adds Grouped and Batched GEMM kernels with blockscaling matching DeepGEMM API",
    Summary, adopts it): any value gives the same bits."""
    p = synth.make_problem("masked", 3, 256, 256, [10, 200, 0], M_max=256, seed=59, device=DEV)
    outs = []
    for em in (0, 1, 128, 1 << 20):
        d = torch.full((p.G, p.M_max, p.N), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        fb.gemm_grouped_masked(p.a, p.sa_mk_view(), p.b, p.sb, d, p.masked_m, em)
        torch.cuda.synchronize()
        assert fb.device_error() == 0
        outs.append(d.view(torch.int16).cpu().numpy())
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    valid, untouched = all_rows(p)
    compare(p, outs[0].view(np.uint16).reshape(-1, p.N), valid, untouched)
