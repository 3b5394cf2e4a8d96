"""Pins of the oracle's fused gate/up epilogue (CPU only).

SiLU(gate) * up ("flydsl mxfp4 a4w4 MoE: bring gemm1/gemm2 to parity with the
HIP backend", section *gemm1*), requantised per (1,128) block with the UE8M0
ceil quantiser of the "Adds Grouped and Batched GEMM kernels with blockscaling
matching DeepGEMM API" page (*DeepGEMM conformance details*).  Each test ties
oracle.silu_mul_quant to something other than itself: hand-derived blocks in
tests/golden/silu_quant_cases.json, closed forms of SiLU, and invariants any
correct quantiser satisfies.  A swapped gate/up, a missing sign, a floor
instead of a ceil scale, truncation instead of rounding or a scale per row
instead of per block fails one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "silu_quant_cases.json")


def _block(spec):
    v = np.full(128, spec["default"], dtype=np.float64)
    for col, val in spec.get("set", []):
        v[col] = val
    return v


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_derived_blocks(oracle_mod, case):
    acc = np.concatenate([_block(case["gate"]), _block(case["up"])])[None, :]
    r = oracle.silu_mul_quant(acc)
    assert r["s"][0, 0] == np.float32(case["scale"])
    for col, code_hex, dequant, h in case["expect"]:
        assert r["q"][0, col] == int(code_hex, 16), (col, hex(r["q"][0, col]))
        assert oracle.e4m3_decode(r["q"][0, col]) * float(r["s"][0, 0]) == dequant
        assert math.isclose(r["h"][0, col], h, rel_tol=1e-14, abs_tol=0.0)


def test_silu_closed_forms(oracle_mod):
    g = np.array([0.0, 1.0, -1.0, 40.0, -40.0, 3.5] + [0.0] * 122)
    u = np.ones(128)
    h = oracle.silu_mul_quant(np.concatenate([g, u])[None, :])["h"][0]
    assert h[0] == 0.0
    assert math.isclose(h[1], 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)   # 0.7310585786...
    assert math.isclose(h[2], -1.0 / (1.0 + math.e), rel_tol=1e-15)
    assert h[3] == 40.0                                  # e^-40 vanishes against 1
    assert abs(h[4]) < 1e-15
    # silu(x) - silu(-x) = x  (x e^x/(1+e^x) + x/(1+e^x) = x)
    gg = np.linspace(-9, 9, 128)
    hp = oracle.silu_mul_quant(np.concatenate([gg, u])[None, :])["h"][0]
    hm = oracle.silu_mul_quant(np.concatenate([-gg, u])[None, :])["h"][0]
    assert np.allclose(hp - hm, gg, rtol=0, atol=1e-13)


def test_gate_and_up_are_not_interchangeable(oracle_mod):
    g = np.full(128, -2.0)
    u = np.full(128, 3.0)
    h1 = oracle.silu_mul_quant(np.concatenate([g, u])[None, :])["h"][0, 0]
    h2 = oracle.silu_mul_quant(np.concatenate([u, g])[None, :])["h"][0, 0]
    assert math.isclose(h1, -6.0 / (1.0 + math.exp(2.0)), rel_tol=1e-14)
    assert math.isclose(h2, -6.0 / (1.0 + math.exp(-3.0)), rel_tol=1e-14)


def _spacing(v):
    """Distance between neighbouring E4M3 values around |v| (subnormal step below 2^-6)."""
    av = np.abs(v)
    e = np.floor(np.log2(np.maximum(av, 2.0 ** -6)))
    return 2.0 ** (e - 3)


def test_quantiser_invariants_on_random_blocks(oracle_mod):
    rng = np.random.default_rng(11)
    rows, i_out = 64, 512
    # accumulator magnitudes of a K = 7168 contraction of unit-variance data
    acc = rng.normal(0.0, 85.0, size=(rows, 2 * i_out))
    acc[3, :] = 0.0                                        # an all-zero row
    acc[5, i_out:i_out + 128] *= 1e-7                      # a tiny block
    r = oracle.silu_mul_quant(acc)
    h, q, s = r["h"], r["q"], r["s"].astype(np.float64)
    # per-block scales: powers of two, ceil of amax/448 (amax floored at 1e-4)
    mant, _ = np.frexp(s)
    assert np.all(mant == 0.5)
    amax = np.maximum(np.abs(h).reshape(rows, -1, 128).max(axis=2), 1e-4)
    t = (amax.astype(np.float32) / np.float32(448.0)).astype(np.float64)
    assert np.all(t <= s) and np.all(s < 2 * t)
    # every scaled value is representable range, error at most half a spacing
    sfull = np.repeat(s, 128, axis=1)
    x = (h.astype(np.float32).astype(np.float64)) / sfull
    assert np.all(np.abs(x) <= 448.0)
    deq = oracle.e4m3_decode(q)
    assert np.all(np.abs(deq - x) <= 0.5 * _spacing(x) + 1e-12)
    # signs survive wherever the value does not round to zero
    nz = np.abs(x) >= 2.0 ** -9
    assert np.all(np.sign(deq[nz]) == np.sign(x[nz]))
    # the all-zero row quantises to +0 codes
    assert np.all(q[3] == 0)
    # margins are distances, tmargins too
    assert np.all(r["margin"] >= 0) and np.all(r["tmargin"] >= 0) and np.all(r["tmargin"] <= 0.5)


def test_scale_is_per_block_not_per_row(oracle_mod):
    g = np.concatenate([np.full(128, 40.0), np.full(128, 40.0)])
    u = np.concatenate([np.full(128, 1.0), np.full(128, 1.0 / 64)])
    r = oracle.silu_mul_quant(np.concatenate([g, u])[None, :])
    # block 0: h = 40, 40/448 in (2^-4, 2^-3]; block 1: h = 0.625, 0.625/448 in (2^-10, 2^-9]
    assert r["s"][0, 0] == np.float32(0.125) and r["s"][0, 1] == np.float32(2.0 ** -9)
    assert oracle.e4m3_decode(r["q"][0, 0]) == 320.0 and oracle.e4m3_decode(r["q"][0, 128]) == 320.0
