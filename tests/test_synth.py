"""The seeded input recipe (CPU only): the generator's quantiser against the
oracle's independently written E4M3 encoder and ceil_to_ue8m0, and the group
size draws of the named workloads."""
import numpy as np
import torch

import oracle
import synth
from synth.inputs import CONFIGS, SA_KM, SA_MK, draw_group_sizes


def test_quantiser_matches_oracle_encoding(oracle_mod):
    gen = torch.Generator().manual_seed(123)
    x = torch.randn(6, 384, generator=gen) * torch.tensor([1e-3, 1.0, 30.0]).repeat_interleave(128)
    x[0, :128] = 0.0  # an all-zero block takes the amax floor
    q, s = synth.quantize_a_blocks(x)
    xs = x.double().numpy()
    amax = np.maximum(np.abs(x.numpy()).reshape(6, 3, 128).max(axis=2), np.float32(1e-4))
    t = (amax.astype(np.float32) / np.float32(448.0)).astype(np.float64)  # fp32 division
    s_or = oracle.ceil_to_ue8m0(t)
    assert np.array_equal(s.double().numpy(), s_or)
    scaled = xs.reshape(6, 3, 128) / s_or[:, :, None]
    assert np.all(np.abs(scaled) <= 448.0)
    codes = oracle.e4m3_encode(scaled).reshape(6, 384)
    same = (codes == q.numpy()) | (((codes & 0x7F) == 0) & ((q.numpy() & 0x7F) == 0))
    assert same.all()


def test_b_quantiser_blocks_are_128_by_128(oracle_mod):
    gen = torch.Generator().manual_seed(5)
    x = torch.randn(256, 256, generator=gen)
    x[128:, 128:] *= 64.0  # one block much larger
    q, s = synth.quantize_b_blocks(x)
    assert s.shape == (2, 2)
    assert s[1, 1] / s[0, 0] >= 32
    deq = oracle.e4m3_decode(q.numpy()) * np.kron(s.double().numpy(), np.ones((128, 128)))
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 on normals
    big = np.abs(x.numpy()) > 0.05 * np.abs(x.numpy()).max()
    rel = np.abs(deq - x.double().numpy())[big] / np.abs(x.double().numpy())[big]
    assert rel.max() <= 2.0 ** -4 + 1e-12


def test_group_size_draws():
    c3 = draw_group_sizes(CONFIGS["c3_contig_g8_mrand_n7168_k2304"]["sizes"], 8, 3)
    assert len(c3) == 8 and all(100 <= m <= 1024 for m in c3)
    c4 = draw_group_sizes(CONFIGS["c4_masked_g16_mmax1024_n2048_k7168"]["sizes"], 16, 4)
    assert len(c4) == 16 and all(1 <= m <= 512 for m in c4)
    c5 = draw_group_sizes(CONFIGS["c5_contig_g32_dirichlet_n4096_k7168"]["sizes"], 32, 5)
    assert len(c5) == 32 and sum(c5) == 65536
    assert draw_group_sizes(("fixed", 100), 2, 1) == [100, 100]
    # deterministic
    assert c5 == draw_group_sizes(CONFIGS["c5_contig_g32_dirichlet_n4096_k7168"]["sizes"], 32, 5)


def test_contiguous_layout_and_scale_layouts():
    p = synth.make_problem("contiguous", 3, 128, 256, [100, 0, 130], sa_layout=SA_KM, seed=7,
                           tail_rows=5)
    lay = p.grouped_layout.numpy()
    assert p.row_offsets == [0, 128, 128, 384]
    assert lay.size == 389
    assert (lay[:100] == 0).all() and (lay[100:128] == -1).all()
    assert (lay[128:258] == 2).all() and (lay[258:] == -1).all()
    assert p.ld_sa % 4 == 0 and p.sa.shape == (2, p.ld_sa)
    assert torch.equal(p.sa_mk(), p.sa[:, :389].t())
    q = synth.make_problem("contiguous", 3, 128, 256, [100, 0, 130], sa_layout=SA_MK, seed=7,
                           tail_rows=5)
    assert torch.equal(q.a, p.a) and torch.equal(q.sa, p.sa_mk())


def test_masked_problem_shapes():
    p = synth.make_problem("masked", 2, 128, 128, [3, 0], M_max=5, sa_layout=SA_KM, seed=9)
    assert p.a.shape == (2, 5, 128) and p.sa.shape == (2, 1, 8)
    assert p.masked_m.tolist() == [3, 0]
    assert p.group_of_row(2) == (0, 2) and p.group_of_row(3)[0] == -1
    assert p.group_of_row(5)[0] == -1
    v, u = synth.sample_rows(p, per_group=4)
    assert set(v.tolist()) <= {0, 1, 2} and 3 in u.tolist()


def test_sample_rows_cover_group_edges():
    p = synth.make_problem("contiguous", 2, 128, 128, [100, 40], seed=3)
    v, u = synth.sample_rows(p, per_group=8)
    assert {0, 99, 128, 167}.issubset(set(v.tolist()))
    assert {100, 127, 168, 255}.issubset(set(u.tolist()))
    for r in v:
        assert p.group_of_row(int(r))[0] >= 0
    for r in u:
        assert p.group_of_row(int(r))[0] == -1


def test_mxfp4_quantiser_invariants():
    """Reading of the OCP MX conversion: per 32-element block the E8M0 byte is
    floor(log2 amax) - 2 + 127, elements are the nearest E2M1 values of x / scale
    (ties to the even code), saturating at 6."""
    import oracle
    from synth.inputs import quantize_mxfp4

    g = torch.Generator().manual_seed(5)
    x = torch.randn(16, 256, generator=g) * torch.logspace(-3, 3, 16).unsqueeze(1)
    x[3] = 0.0
    packed, sc = quantize_mxfp4(x)
    assert packed.shape == (16, 128) and sc.shape == (16, 8)
    codes = torch.stack([packed & 0xF, packed >> 4], dim=-1).reshape(16, 256).numpy()
    vals = oracle.e2m1_decode(codes)
    scale = np.ldexp(1.0, sc.numpy().astype(np.int64) - 127)
    xb = x.double().numpy().reshape(16, 8, 32)
    amax = np.maximum(np.abs(xb).max(axis=2), 1e-4)
    assert np.array_equal(sc.numpy().astype(np.int64) - 127, np.floor(np.log2(amax)) - 2)
    y = xb / scale[..., None]
    deq = vals.reshape(16, 8, 32)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    # nearest representable magnitude (saturating), compared by distance
    best = np.abs(np.abs(y)[..., None] - grid).min(axis=-1)
    assert np.allclose(np.abs(np.abs(deq) - np.minimum(np.abs(y), 6.0)),
                       np.minimum(best, np.abs(np.minimum(np.abs(y), 6.0) - np.abs(deq))))
    assert np.all(np.abs(np.abs(deq) - np.abs(y)) <= np.maximum(best, np.abs(y) - 6.0) + 1e-12)
    assert np.all((deq == 0) | (np.sign(deq) == np.sign(y)))
    assert np.all(codes[3] == 0)


def test_sample_rows_cover_every_tile_and_all_untouched_rows():
    """Every 128-row tile that holds a valid row contributes a sampled row, and
    every row that must not be written is listed."""
    for p in (synth.make_problem("contiguous", 3, 128, 128, [300, 0, 129], seed=4, tail_rows=20),
              synth.make_problem("masked", 3, 128, 128, [0, 257, 130], M_max=300, seed=5)):
        v, u = synth.sample_rows(p, per_group=2)
        vs = set(v.tolist())
        for r in range(p.rows):
            g, m = p.group_of_row(r)
            if g < 0:
                assert r in set(u.tolist())
        for g, m in enumerate(p.group_sizes):
            base = p.row_offsets[g] if p.variant == "contiguous" else g * p.M_max
            for t0 in range(0, m, 128):
                assert any(base + t0 <= r < base + min(m, t0 + 128) for r in vs), (g, t0)
        assert len(u) == p.rows - p.valid_rows
