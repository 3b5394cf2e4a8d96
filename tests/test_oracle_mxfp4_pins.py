"""Pins of the oracle's MXFP4 (a4w4) grouped GEMM (CPU only).

The operation is the MoE GEMM with both operands in MXFP4 of the page "flydsl
mxfp4 a4w4 MoE: bring gemm1/gemm2 to parity with the HIP backend" (Summary),
with the OCP Microscaling definition of the format: E2M1 elements, one E8M0
scale per 32 consecutive elements along K, two elements per byte (element 2i
in the low nibble).  Pinned against a hand-derived E2M1 table, the E8M0
closed form, exact rationals, the integer matmul and power-of-two scaling; a
swapped nibble order, a scale applied to the wrong block or row, or a dropped
block fails one of them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_values.json")


def test_e2m1_table_hand_derived(oracle_mod):
    want = json.load(open(GOLDEN))["values"]
    got = oracle.e2m1_decode(np.arange(16))
    for code, v in want.items():
        assert got[int(code)] == v and np.signbit(got[int(code)]) == np.signbit(v), code


def test_e8m0_closed_form(oracle_mod):
    e = np.arange(255)
    assert np.array_equal(oracle.e8m0_decode(e), np.ldexp(1.0, e - 127))
    assert np.isnan(oracle.e8m0_decode([255])[0])


def _pack(codes):
    """[..., K] 4-bit codes -> [..., K/2] bytes, element 2i in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _brute(a_codes, sa, b_codes, sb, layout):
    table = [Fraction(float(v)) for v in oracle.e2m1_decode(np.arange(16))]
    out = {}
    for r, g in enumerate(layout):
        if g < 0:
            continue
        row = []
        for n in range(b_codes.shape[1]):
            tot = Fraction(0)
            for j in range(a_codes.shape[1] // 32):
                s = Fraction(2) ** (int(sa[r, j]) - 127) * Fraction(2) ** (int(sb[g, n, j]) - 127)
                dot = sum(table[a_codes[r, k]] * table[b_codes[g, n, k]]
                          for k in range(32 * j, 32 * j + 32))
                tot += s * dot
            row.append(tot)
        out[r] = row
    return out


def test_contiguous_matches_exact_rationals(oracle_mod):
    rng = np.random.default_rng(31)
    layout = np.array([0, 0, -1, 1, 1, 1, -1, -1], dtype=np.int32)
    K, N, G = 96, 6, 2
    a = rng.integers(0, 16, (8, K)).astype(np.uint8)
    b = rng.integers(0, 16, (G, N, K)).astype(np.uint8)
    sa = rng.integers(117, 138, (8, K // 32)).astype(np.uint8)
    sb = rng.integers(117, 138, (G, N, K // 32)).astype(np.uint8)
    acc, valid, rows = oracle.mxfp4_contiguous(_pack(a), sa, _pack(b), sb, layout)
    brute = _brute(a, sa, b, sb, layout)
    assert valid.tolist() == [g >= 0 for g in layout]
    for i, r in enumerate(rows):
        if valid[i]:
            assert [Fraction(float(x)) for x in acc[i]] == brute[r]
        else:
            assert np.isnan(acc[i]).all()


def test_integer_matmul_special_case(oracle_mod):
    """Unit scales (E8M0 127) and integer-valued elements: the integer matmul."""
    rng = np.random.default_rng(32)
    ints = {0: 0, 2: 1, 4: 2, 5: 3, 6: 4, 7: 6, 10: -1, 12: -2, 13: -3, 15: -6}
    codes = np.array(list(ints), dtype=np.uint8)
    K, N = 128, 4
    a = rng.choice(codes, (3, K))
    b = rng.choice(codes, (1, N, K))
    val = np.vectorize(ints.get)
    want = val(a).astype(np.int64) @ val(b[0]).astype(np.int64).T
    sa = np.full((3, K // 32), 127, np.uint8)
    sb = np.full((1, N, K // 32), 127, np.uint8)
    acc, _, _ = oracle.mxfp4_contiguous(_pack(a), sa, _pack(b), sb, np.zeros(3, np.int32))
    assert np.array_equal(acc, want.astype(np.float64))


def test_nibble_order_and_block_scale_index(oracle_mod):
    """B row 0 holds 1.0 at element 0 only (the low nibble of byte 0), row 1 at
    element 33 only (second scale block); A's second block scale is 2^3."""
    K = 64
    b = np.zeros((1, 2, K), np.uint8)
    b[0, 0, 0] = 2
    b[0, 1, 33] = 2
    sa = np.array([[127, 130]], np.uint8)
    sb = np.full((1, 2, 2), 127, np.uint8)

    def run(pos, code):
        a = np.zeros((1, K), np.uint8)
        a[0, pos] = code
        acc, _, _ = oracle.mxfp4_contiguous(_pack(a), sa, _pack(b), sb, np.zeros(1, np.int32))
        return acc.tolist()

    assert run(0, 2) == [[1.0, 0.0]]     # element 0 (low nibble) meets B[0, 0]
    assert run(1, 7) == [[0.0, 0.0]]     # element 1 (high nibble) meets nothing
    assert run(33, 2) == [[0.0, 8.0]]    # element 33: block 1 of A (2^3) times B[1, 33]
    assert run(32, 2) == [[0.0, 0.0]]


def test_masked_full_equals_contiguous(oracle_mod):
    rng = np.random.default_rng(33)
    G, M, N, K = 2, 5, 8, 64
    a = rng.integers(0, 256, (G, M, K // 2)).astype(np.uint8)
    sa = rng.integers(120, 134, (G, M, K // 32)).astype(np.uint8)
    b = rng.integers(0, 256, (G, N, K // 2)).astype(np.uint8)
    sb = rng.integers(120, 134, (G, N, K // 32)).astype(np.uint8)
    accm, vm, _ = oracle.mxfp4_masked(a, sa, b, sb, np.array([M, M], np.int32))
    layout = np.repeat(np.arange(G, dtype=np.int32), M)
    accc, vc, _ = oracle.mxfp4_contiguous(a.reshape(G * M, -1), sa.reshape(G * M, -1), b, sb,
                                          layout)
    assert vm.all() and vc.all() and np.array_equal(accm, accc)
    accp, vp, _ = oracle.mxfp4_masked(a, sa, b, sb, np.array([2, 0], np.int32))
    assert vp.tolist() == [True, True, False, False, False] + [False] * 5
