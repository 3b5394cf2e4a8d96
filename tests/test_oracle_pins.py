"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to an independent authority: a library
conversion routine (torch / numpy), exact rational arithmetic (brute force
with fractions.Fraction), a textbook special case (integer matmul), a closed
form, or a hand-derived case under tests/golden/.  The chosen inputs make the
plausible mistakes fail: a dropped K-block, a wrong scale index (n/128 vs kb,
transposed activation scales), a transposed B operand, a wrong group, a sign
error or a wrong rounding rule.

The definition being pinned is the one on the "Adds Grouped and Batched GEMM
kernels with blockscaling matching DeepGEMM API" page (FlyDSL PR #433),
sections *Summary* and *DeepGEMM conformance details*.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.inputs import SA_KM, SA_MK

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ element codecs
def test_e4m3_decode_exhaustive_vs_torch(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    # format facts: max 448, min subnormal 2^-9, exactly two NaN codes
    assert np.nanmax(ours) == 448.0
    assert ours[1] == 2.0 ** -9
    assert np.isnan(ours).sum() == 2


def _e4m3_positive_values():
    return np.array(sorted(v for v in oracle.e4m3_table()[:127]), dtype=np.float64)


def test_e4m3_encode_vs_torch_ties_and_samples(oracle_mod):
    vals = _e4m3_positive_values()
    mids = (vals[:-1] + vals[1:]) / 2  # exact ties, representable in fp32
    rng = np.random.default_rng(0)
    rand = rng.uniform(-448, 448, size=4000)
    tiny = rng.uniform(-2 ** -6, 2 ** -6, size=1000)
    xs = np.concatenate([vals, -vals, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                         rand, tiny]).astype(np.float32).astype(np.float64)
    ours = oracle.e4m3_encode(xs)
    ref = torch.from_numpy(xs.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # +-0 may differ only in sign for values that round to zero
    same = (ours == ref) | ((ours & 0x7F) == 0) & ((ref & 0x7F) == 0)
    assert same.all(), xs[~same][:10]


def test_e4m3_encode_saturates(oracle_mod):
    assert oracle.e4m3_encode([448.0, 449.0, 1e6, -1e6]).tolist() == [0x7E, 0x7E, 0x7E, 0xFE]


def test_ceil_to_ue8m0_powers_of_two_exhaustive(oracle_mod):
    ts, want = [], []
    for e in range(-125, 127):
        t = np.float32(2.0 ** e)
        ts += [t, np.nextafter(t, np.float32(np.inf)), np.nextafter(t, np.float32(0))]
        want += [2.0 ** e, 2.0 ** (e + 1), 2.0 ** e]
    ts = np.array(ts, dtype=np.float32)
    got = oracle.ceil_to_ue8m0(ts.astype(np.float64))
    assert np.array_equal(got, np.array(want))
    # the generator's bit-level version agrees value for value
    gen = synth.ceil_to_ue8m0_f32(torch.from_numpy(ts)).double().numpy()
    assert np.array_equal(gen, got)


def test_ceil_to_ue8m0_properties(oracle_mod):
    rng = np.random.default_rng(1)
    t = (rng.uniform(0.5, 1.0, 3000) * 2.0 ** rng.integers(-30, 30, 3000)).astype(np.float32)
    s = oracle.ceil_to_ue8m0(t.astype(np.float64))
    m, _ = np.frexp(s)
    assert np.all(m == 0.5)                       # a power of two
    assert np.all(s >= t) and np.all(s / 2 < t)   # the smallest such
    gen = synth.ceil_to_ue8m0_f32(torch.from_numpy(t)).double().numpy()
    assert np.array_equal(gen, s)


def test_round_bf16_vs_torch(oracle_mod):
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # explicit ties: halfway between two bf16 values, both parities
    base = rng.integers(0, 2 ** 16, size=2000, dtype=np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1e-45, 3.4e38])])
    ours = oracle.round_out(x.astype(np.float64), oracle.OUT_BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.uint16).numpy() if hasattr(torch, "uint16") \
        else torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_f16_vs_numpy(oracle_mod):
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(50000) * 100.0,
        rng.uniform(-6.5e4, 6.5e4, 20000),
        rng.uniform(-1e-4, 1e-4, 20000),            # subnormal range
        np.float16(rng.standard_normal(5000)).astype(np.float64),  # exact f16 values
        [65504.0, 65519.99, 65520.0, -65520.0, 2 ** -24, 2 ** -25, 3 * 2 ** -26],
    ])
    # ties: midpoints between adjacent f16 values
    h = np.float16(rng.standard_normal(5000) * 10).astype(np.float64)
    up = np.nextafter(np.float16(h), np.float16(np.inf)).astype(np.float64)
    x = np.concatenate([x, (h + up) / 2])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    ours = oracle.round_out(x, oracle.OUT_F16)
    assert np.array_equal(ours, ref)


def test_calc_diff_closed_forms(oracle_mod):
    rng = np.random.default_rng(4)
    x = rng.standard_normal(1000)
    assert oracle.calc_diff(x, x) == 0.0
    assert math.isclose(oracle.calc_diff(x, -x), 2.0, rel_tol=0, abs_tol=1e-15)
    assert math.isclose(oracle.calc_diff(x, np.zeros_like(x)), 1.0, abs_tol=1e-15)
    assert math.isclose(oracle.calc_diff(x, 2 * x), 1 - 4 / 5, abs_tol=1e-15)
    assert oracle.calc_diff(np.zeros(4), np.zeros(4)) == 0.0
    y = rng.standard_normal(1000)
    assert math.isclose(oracle.calc_diff(x, y), oracle.calc_diff(y, x), abs_tol=1e-15)


# ------------------------------------------------------------------ block arithmetic
def test_block_dot_exact_vs_fractions(oracle_mod):
    rng = np.random.default_rng(5)
    table = oracle.e4m3_table()
    finite = np.array([c for c in range(256) if not np.isnan(table[c])], dtype=np.uint8)
    for _ in range(20):
        x = rng.choice(finite, 128)
        y = rng.choice(finite, 128)
        exact = sum(Fraction(float(table[a])) * Fraction(float(table[b])) for a, b in zip(x, y))
        assert Fraction(oracle.block_dot_exact(x, y)) == exact


def _brute_contiguous(a, sa, sa_layout, b, sb, layout):
    """Dequantise-then-matmul with exact rationals (the reference style of the
    page's *Notes for reviewers*), row by row."""
    table = oracle.e4m3_table()
    m_sum, k = a.shape
    G, n, _ = b.shape
    out = {}
    for r in range(m_sum):
        g = int(layout[r])
        if g < 0:
            continue
        row = []
        for j in range(n):
            tot = Fraction(0)
            for kk in range(k):
                s_a = sa[r, kk // 128] if sa_layout == SA_MK else sa[kk // 128, r]
                s_b = sb[g, j // 128, kk // 128]
                tot += (Fraction(float(table[a[r, kk]])) * Fraction(float(s_a))
                        * Fraction(float(table[b[g, j, kk]])) * Fraction(float(s_b)))
            row.append(tot)
        out[r] = row
    return out


def _random_small_problem(rng, G, rows_per_group, N, K, pad_to=4, exp_range=(-12, 4)):
    """Tiny problem with random codes, random power-of-two scales and -1 rows."""
    table = oracle.e4m3_table()
    finite = np.array([c for c in range(256) if not np.isnan(table[c])], dtype=np.uint8)
    layout = []
    for g, m in enumerate(rows_per_group):
        layout += [g] * m + [-1] * (-m % pad_to)
    layout = np.array(layout, dtype=np.int32)
    M = layout.size
    a = rng.choice(finite, (M, K))
    b = rng.choice(finite, (G, N, K))
    sa = (2.0 ** rng.integers(*exp_range, (M, K // 128))).astype(np.float32)
    sb = (2.0 ** rng.integers(*exp_range, (G, N // 128, K // 128))).astype(np.float32)
    return a, sa, b, sb, layout


@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM])
def test_contiguous_matches_exact_rationals(oracle_mod, sa_layout):
    """Wide scale spread (2^-12..2^3), two K-blocks: each block term is exact in
    fp64 and the oracle adds two exact terms once, so its result must be the
    correctly rounded exact value, element for element."""
    rng = np.random.default_rng(6 + sa_layout)
    # N = 256 so that the n/128 scale index takes two values; K = 256: two K-blocks
    a, sa_mk, b, sb, layout = _random_small_problem(rng, 3, [2, 1, 3], 256, 256)
    sa = sa_mk if sa_layout == SA_MK else np.ascontiguousarray(sa_mk.T)
    acc, valid, rows = oracle.grouped_contiguous(a, sa, sa_layout, b, sb, layout)
    brute = _brute_contiguous(a, sa, sa_layout, b, sb, layout)
    assert set(rows[valid].tolist()) == set(brute)
    for i, r in enumerate(rows):
        if not valid[i]:
            assert layout[r] == -1 and np.isnan(acc[i]).all()
            continue
        assert all(float(acc[i, j]) == float(brute[r][j]) for j in range(acc.shape[1]))


def test_contiguous_with_arbitrary_fp32_scales_vs_exact_rationals(oracle_mod):
    """Scales that are not powers of two (the inputs of the software-promotion
    path): the oracle's fp64 result is within a few fp64 ulps of the exact
    rational value (no exactness argument holds any more, but nothing coarser
    than fp64 rounding may appear)."""
    rng = np.random.default_rng(21)
    a, sa, b, sb, layout = _random_small_problem(rng, 2, [3, 2], 256, 384, exp_range=(-9, -4))
    sa = (sa * rng.uniform(1.0, 2.0, sa.shape)).astype(np.float32)
    sb = (sb * rng.uniform(1.0, 2.0, sb.shape)).astype(np.float32)
    assert np.any(np.frexp(sa)[0] != 0.5) and np.any(np.frexp(sb)[0] != 0.5)
    acc, valid, rows = oracle.grouped_contiguous(a, sa, SA_MK, b, sb, layout)
    brute = _brute_contiguous(a, sa, SA_MK, b, sb, layout)
    # the same sums over |terms| (sign bits cleared) bound the rounding of the fp64 ones
    mags = _brute_contiguous(a & 0x7F, sa, SA_MK, b & 0x7F, sb, layout)
    for i, r in enumerate(rows):
        if not valid[i]:
            continue
        for j in range(acc.shape[1]):
            err = abs(Fraction(float(acc[i, j])) - brute[r][j])
            assert err <= mags[r][j] * Fraction(1, 2 ** 48)


def test_contiguous_exact_with_realistic_scale_spread(oracle_mod):
    """Scales within 2^-9..2^-5 (the spread ceil_to_ue8m0 gives N(0,1) data) and
    four K-blocks: the fp64 sum is the exact rational value, bit for bit."""
    rng = np.random.default_rng(13)
    a, sa, b, sb, layout = _random_small_problem(rng, 2, [2, 2], 128, 512, exp_range=(-9, -4))
    acc, valid, rows = oracle.grouped_contiguous(a, sa, SA_MK, b, sb, layout)
    brute = _brute_contiguous(a, sa, SA_MK, b, sb, layout)
    for i, r in enumerate(rows):
        if valid[i]:
            assert all(Fraction(float(acc[i, j])) == brute[r][j] for j in range(acc.shape[1]))


def test_integer_matmul_special_case(oracle_mod):
    """G=1, all scales 1, codes of small integers: D is the integer matmul."""
    rng = np.random.default_rng(7)
    ints = np.arange(-4, 5)
    enc = {v: int(oracle.e4m3_encode([float(v)])[0]) for v in ints}
    ai = rng.choice(ints, (5, 256))
    bi = rng.choice(ints, (1, 128, 256))
    a = np.vectorize(enc.get)(ai).astype(np.uint8)
    b = np.vectorize(enc.get)(bi).astype(np.uint8)
    sa = np.ones((5, 2), np.float32)
    sb = np.ones((1, 1, 2), np.float32)
    acc, valid, _ = oracle.grouped_contiguous(a, sa, SA_MK, b, sb, np.zeros(5, np.int32))
    want = ai.astype(np.int64) @ bi[0].astype(np.int64).T
    assert valid.all() and np.array_equal(acc, want.astype(np.float64))
    # |D| <= 256 here would be exact in bf16 as well; check the rounding keeps it
    small = np.abs(want) <= 256
    bits = oracle.round_out(acc, oracle.OUT_BF16)
    assert np.array_equal(oracle.bits_to_float(bits, oracle.OUT_BF16)[small], acc[small])


def test_power_of_two_scale_exactness(oracle_mod):
    """Only K-block 1 is non-zero; scaling sa[r,1] or sb[g,nb,1] by 2^j scales the
    output of exactly the affected rows / 128-column blocks by 2^j."""
    rng = np.random.default_rng(8)
    a, sa, b, sb, _ = _random_small_problem(rng, 1, [4], 256, 256)
    a[:, :128] = 0
    layout = np.zeros(4, np.int32)
    base, _, _ = oracle.grouped_contiguous(a, sa, SA_MK, b, sb, layout)
    sa2 = sa.copy()
    sa2[2, 1] *= 2.0 ** 5
    sa2[1, 0] *= 2.0 ** 9  # block 0 is all zero: no effect
    got, _, _ = oracle.grouped_contiguous(a, sa2, SA_MK, b, sb, layout)
    want = base.copy()
    want[2] *= 2.0 ** 5
    assert np.array_equal(got, want)
    sb2 = sb.copy()
    sb2[0, 1, 1] *= 2.0 ** -3  # columns 128..255 only
    got, _, _ = oracle.grouped_contiguous(a, sa, SA_MK, b, sb2, layout)
    want = base.copy()
    want[:, 128:] *= 2.0 ** -3
    assert np.array_equal(got, want)


def test_masked_full_equals_contiguous(oracle_mod):
    rng = np.random.default_rng(9)
    G, M, N, K = 3, 5, 128, 256
    a, sa, b, sb, layout = _random_small_problem(rng, G, [M] * G, N, K, pad_to=1)
    acc_c, valid_c, _ = oracle.grouped_contiguous(a, sa, SA_MK, b, sb, layout)
    mm = np.full(G, M, np.int32)
    acc_m, valid_m, _ = oracle.grouped_masked(a.reshape(G, M, K), sa.reshape(G, M, 2), SA_MK,
                                               b, sb, mm)
    assert valid_c.all() and valid_m.all()
    assert np.array_equal(acc_c, acc_m)
    # transposed per-group scale layout gives the same numbers
    sa_km = np.ascontiguousarray(sa.reshape(G, M, 2).transpose(0, 2, 1))
    acc_t, _, _ = oracle.grouped_masked(a.reshape(G, M, K), sa_km, SA_KM, b, sb, mm)
    assert np.array_equal(acc_m, acc_t)


def test_masked_rows_and_padding_rows_produce_nothing(oracle_mod):
    rng = np.random.default_rng(10)
    G, M, N, K = 2, 4, 128, 128
    a, sa, b, sb, _ = _random_small_problem(rng, G, [M] * G, N, K, pad_to=1)
    mm = np.array([3, 0], np.int32)
    acc, valid, rows = oracle.grouped_masked(a.reshape(G, M, K), sa.reshape(G, M, 1), SA_MK,
                                             b, sb, mm)
    assert valid.tolist() == [True, True, True, False, False, False, False, False]
    assert np.isnan(acc[~valid]).all() and np.isfinite(acc[valid]).all()


def test_group_permutation_permutes_outputs(oracle_mod):
    rng = np.random.default_rng(11)
    a, sa, b, sb, layout = _random_small_problem(rng, 3, [2, 3, 1], 128, 256)
    perm = np.array([2, 0, 1])          # new group id of old group g
    inv = np.argsort(perm)
    layout2 = np.where(layout >= 0, perm[np.maximum(layout, 0)], -1).astype(np.int32)
    acc1, v1, _ = oracle.grouped_contiguous(a, sa, SA_MK, b, sb, layout)
    acc2, v2, _ = oracle.grouped_contiguous(a, sa, SA_MK, b[inv], sb[inv], layout2)
    assert np.array_equal(v1, v2)
    assert np.array_equal(acc1[v1], acc2[v2])


def test_transposed_b_would_be_caught(oracle_mod):
    """Sanity of the pins themselves: a problem where using B[g,k,n] instead of
    B[g,n,k] changes the answer (square blocks, non-symmetric data)."""
    rng = np.random.default_rng(12)
    a, sa, b, sb, layout = _random_small_problem(rng, 1, [2], 128, 128, pad_to=1)
    acc, _, _ = oracle.grouped_contiguous(a, sa, SA_MK, b, sb, layout)
    bt = np.ascontiguousarray(b.transpose(0, 2, 1))
    acc_t, _, _ = oracle.grouped_contiguous(a, sa, SA_MK, bt, sb, layout)
    assert not np.array_equal(acc, acc_t)


# ------------------------------------------------------------------ hand-derived golden cases
def _load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _load_golden("hand_cases.json")["cases"], ids=lambda c: c["name"])
def test_hand_cases(oracle_mod, case):
    def fill(spec, shape):
        arr = np.empty(shape, dtype=np.uint8)
        arr[...] = spec["default"]
        for ranges, code in spec.get("fill", []):
            arr[tuple(slice(lo, hi) for lo, hi in ranges)] = code
        return arr

    K, N, G = case["K"], case["N"], case["G"]
    b = fill(case["b_codes"], (G, N, K))
    sb = np.array(case["scale_b"], np.float32).reshape(G, N // 128, K // 128)
    if case["variant"] == "contiguous":
        M = len(case["grouped_layout"])
        a = fill(case["a_codes"], (M, K))
        sa = np.array(case["scale_a"], np.float32).reshape(M, K // 128)
        acc, valid, _ = oracle.grouped_contiguous(a, sa, SA_MK, b, sb,
                                                  np.array(case["grouped_layout"], np.int32))
    else:
        Mx = case["M_max"]
        a = fill(case["a_codes"], (G, Mx, K))
        sa = np.array(case["scale_a"], np.float32).reshape(G, Mx, K // 128)
        acc, valid, _ = oracle.grouped_masked(a, sa, SA_MK, b, sb,
                                              np.array(case["masked_m"], np.int32))
    assert valid.tolist() == case["valid"]
    for r, expect in case["expect_rows"].items():
        r = int(r)
        bits = oracle.round_out(acc[r], case["out_dtype"])
        for lo, hi, value, hexbits in expect["segments"]:
            assert np.all(acc[r, lo:hi] == value), (r, acc[r, lo:hi][:4])
            assert np.all(bits[lo:hi] == int(hexbits, 16)), (r, hex(int(bits[lo])))


# ------------------------------------------------------------------ the pages' end-to-end convention
@pytest.mark.parametrize("sa_layout", [SA_MK, SA_KM])
def test_config1_within_fp32_reference(oracle_mod, sa_layout):
    """calc_diff(oracle, a_f32 @ b_f32.T) <= 1e-3 on valid rows (the threshold and
    reference convention of the page's *DeepGEMM conformance details*)."""
    p = synth.make_problem("contiguous", 2, 256, 256, [100, 100], sa_layout=sa_layout, seed=1)
    acc, valid, rows = oracle.grouped_contiguous(p.a.numpy(), p.sa.numpy(), p.sa_layout,
                                                 p.b.numpy(), p.sb.numpy(),
                                                 p.grouped_layout.numpy(), ld_sa=p.ld_sa)
    ref = []
    for g in range(p.G):
        ref.append((p.regen_a_f32(g).double() @ p.regen_b_f32(g).double().T)[: p.group_sizes[g]])
    ref = torch.cat(ref).numpy()
    d = oracle.calc_diff(acc[valid], ref)
    assert 1e-5 < d <= 1e-3  # quantisation error is present but within budget


def test_deepseek_shape_within_fp32_reference(oracle_mod):
    """Same convention at the N=2048, K=7168 expert shape on a few rows."""
    p = synth.make_problem("contiguous", 2, 2048, 7168, [3, 2], sa_layout=SA_KM, seed=21,
                           pad_multiple=4)
    acc, valid, rows = oracle.grouped_contiguous(p.a.numpy(), p.sa.numpy(), p.sa_layout,
                                                 p.b.numpy(), p.sb.numpy(),
                                                 p.grouped_layout.numpy(), ld_sa=p.ld_sa)
    ref = []
    for g in range(p.G):
        ref.append((p.regen_a_f32(g).double() @ p.regen_b_f32(g).double().T)[: p.group_sizes[g]])
    ref = torch.cat(ref).numpy()
    assert oracle.calc_diff(acc[valid], ref) <= 1e-3
