"""Seeded workload generator and UE8M0 block quantiser (input recipe only).

Shapes of the named workloads follow the coverage named on the FlyDSL PR #433
page ("Adds Grouped and Batched GEMM kernels with blockscaling matching
DeepGEMM API", *Test plan*): 1-8 (and 16/32) groups, m_per_group from the
unaligned 100 up to 1024, the DeepSeek-V3 expert shapes N=2048/K=7168 and
N=7168/K=2304, bf16 and f16 outputs; plus the dense 4096 x 4096 x 16384 shape of the
FP8 figure on the "[Kernel][MI350] Add cache-aware 8-wave BF16/FP16 GEMM" page
(*Performance*), run as a single group.

All draws are seeded.  Group sizes come from numpy's PCG64 (identical on every
platform); the N(0,1) data comes from a torch generator on the chosen device,
one sub-seed per (tensor, group) so that any group can be regenerated alone
without holding a large workload's fp32 data in memory.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

SA_MK = 0  # scale_a [rows, K/128]
SA_KM = 1  # scale_a transposed [K/128, ld_sa] (per group for the masked variant)
OUT_BF16 = 0
OUT_F16 = 1
E4M3_MAX = 448.0
AMAX_FLOOR = 1e-4

# name -> parameters; "sizes" names the group-size draw.
CONFIGS: Dict[str, dict] = {
    # contiguous, G=2, 100 rows per expert padded to 128 with -1 rows
    "c1_contig_g2_m100_n256_k256": dict(
        variant="contiguous", G=2, N=256, K=256, out=OUT_BF16, sa_layout=SA_MK,
        sizes=("fixed", 100), seed=1),
    # contiguous, G=8, 1024 rows per expert, activation scales transposed
    "c2_contig_g8_m1024_n2048_k7168": dict(
        variant="contiguous", G=8, N=2048, K=7168, out=OUT_BF16, sa_layout=SA_KM,
        sizes=("fixed", 1024), seed=2),
    # contiguous, G=8, m_g ~ U[100, 1024] padded to 128, f16 output
    "c3_contig_g8_mrand_n7168_k2304": dict(
        variant="contiguous", G=8, N=7168, K=2304, out=OUT_F16, sa_layout=SA_MK,
        sizes=("uniform", 100, 1024), seed=3),
    # masked decode, G=16, M_max=1024, masked_m ~ U[1, 512]
    "c4_masked_g16_mmax1024_n2048_k7168": dict(
        variant="masked", G=16, N=2048, K=7168, out=OUT_BF16, sa_layout=SA_KM,
        M_max=1024, sizes=("uniform", 1, 512), seed=4),
    # contiguous prefill, G=32, Dirichlet(0.5) routing of 65536 rows, padded to 128
    "c5_contig_g32_dirichlet_n4096_k7168": dict(
        variant="contiguous", G=32, N=4096, K=7168, out=OUT_BF16, sa_layout=SA_MK,
        sizes=("dirichlet", 0.5, 65536), seed=5),
    # dense GEMM as the G = 1 case of the contiguous layout: 4096 x 4096 x 16384, the
    # FP8 shape whose throughput the pages publish (there with row scales, on other
    # hardware; here block-scaled like every other workload)
    "c6_dense_g1_m4096_n4096_k16384": dict(
        variant="contiguous", G=1, N=4096, K=16384, out=OUT_BF16, sa_layout=SA_MK,
        sizes=("fixed", 4096), seed=6),
    # the first MoE GEMM with its fused epilogue: B holds each expert's gate rows
    # [0, 2048) and up rows [2048, 4096) (DeepSeek-V3 expert shape, hidden 7168,
    # intermediate 2048); the output is SiLU(gate) * up requantised to E4M3 with
    # (1,128) UE8M0 scales in the activation-scale layout named by sa_layout
    "c7_swiglu_contig_g8_m1024_n4096_k7168": dict(
        variant="contiguous", G=8, N=4096, K=7168, out=OUT_BF16, sa_layout=SA_KM,
        sizes=("fixed", 1024), seed=7, epilogue="silu_mul_quant"),
    # workload 2's shape with arbitrary fp32 block scales (amax / 448, not rounded to a
    # power of two), run by the software-promotion kernel
    "c8_fp32scales_contig_g8_m1024_n2048_k7168": dict(
        variant="contiguous", G=8, N=2048, K=7168, out=OUT_BF16, sa_layout=SA_KM,
        sizes=("fixed", 1024), seed=8, scale_kind="fp32"),
    # workload 2's shape with both operands in MXFP4 (E2M1, E8M0 per 32 elements)
    "c9_mxfp4_contig_g8_m1024_n2048_k7168": dict(
        variant="contiguous", G=8, N=2048, K=7168, out=OUT_BF16, sa_layout=SA_MK,
        sizes=("fixed", 1024), seed=9, scale_kind="mxfp4"),
    # workload 2's shape with N not a multiple of 256 (7.5 column tiles of 256)
    "c10_contig_g8_m1024_n1920_k7168": dict(
        variant="contiguous", G=8, N=1920, K=7168, out=OUT_BF16, sa_layout=SA_KM,
        sizes=("fixed", 1024), seed=10),
}


def ceil_to_ue8m0_f32(t: torch.Tensor) -> torch.Tensor:
    """Smallest power of two >= t for positive normal fp32 t, from the fp32 bits.

    A power of two has a zero mantissa field and is kept; any other value has
    its exponent field raised by one and its mantissa cleared.
    """
    if t.dtype != torch.float32:
        raise TypeError("ceil_to_ue8m0_f32 takes fp32")
    bits = t.contiguous().view(torch.int32)
    expo = (bits >> 23) & 0xFF
    mant = bits & 0x7FFFFF
    expo = expo + (mant != 0).to(torch.int32)
    return (expo << 23).view(torch.float32)


def _block_scale(amax: torch.Tensor, pow2: bool) -> torch.Tensor:
    """amax / 448, rounded up to a power of two (UE8M0) unless pow2 is False."""
    t = amax / E4M3_MAX
    return ceil_to_ue8m0_f32(t) if pow2 else t


def quantize_a_blocks(x: torch.Tensor, pow2: bool = True):
    """(1,128) blocks of a [R, K] fp32 matrix -> (e4m3 codes uint8 [R,K], fp32 scales [R,K/128]).

    pow2=False keeps the plain fp32 scale amax / 448 (arbitrary fp32 scales)."""
    r, k = x.shape
    if k % 128:
        raise ValueError("K must be a multiple of 128")
    xb = x.float().reshape(r, k // 128, 128)
    amax = xb.abs().amax(dim=2).clamp(min=AMAX_FLOOR)
    s = _block_scale(amax, pow2)
    q = (xb / s.unsqueeze(2)).to(torch.float8_e4m3fn).view(torch.uint8).reshape(r, k)
    return q, s


def quantize_b_blocks(x: torch.Tensor, pow2: bool = True):
    """(128,128) blocks of an [N, K] fp32 matrix -> (codes uint8 [N,K], scales [N/128,K/128])."""
    n, k = x.shape
    if k % 128 or n % 128:
        raise ValueError("N and K must be multiples of 128")
    xb = x.float().reshape(n // 128, 128, k // 128, 128)
    amax = xb.abs().amax(dim=(1, 3)).clamp(min=AMAX_FLOOR)
    s = _block_scale(amax, pow2)
    q = (xb / s[:, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, k)
    return q, s


# E2M1 rounding boundaries: midpoints between neighbouring magnitudes
# 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7)
_E2M1_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def quantize_mxfp4(x: torch.Tensor):
    """[R, K] fp32 -> (packed E2M1 codes uint8 [R, K/2], E8M0 scale bytes uint8 [R, K/32]).

    Reading of the OCP Microscaling conversion for MXFP4: per block of 32
    elements along K the shared exponent is floor(log2 amax) - 2 (2 being the
    largest E2M1 exponent; amax at least 1e-4), the scale is 2^that, and each
    element x / scale goes to the nearest E2M1 value, ties to the even
    mantissa, magnitudes above 6 saturating to 6.  Element 2i lands in the low
    nibble of byte i.
    """
    r, k = x.shape
    if k % 32:
        raise ValueError("K must be a multiple of 32")
    xb = x.float().reshape(r, k // 32, 32)
    amax = xb.abs().amax(dim=2).clamp(min=AMAX_FLOOR).contiguous()
    e = ((amax.view(torch.int32) >> 23) & 0xFF) - 127        # floor(log2 amax), amax normal
    se = (e - 2).clamp(-127, 127)
    scale = torch.ldexp(torch.ones_like(amax), se)
    y = xb / scale.unsqueeze(2)                               # exact: power-of-two scale
    mag = y.abs()
    mids = torch.tensor(_E2M1_MIDS, dtype=torch.float32, device=x.device)
    idx = torch.bucketize(mag, mids)                          # mids[i-1] < mag <= mids[i] -> i
    tie = (mag == mids[idx.clamp(max=len(_E2M1_MIDS) - 1)]) & (idx % 2 == 1)
    idx = idx + tie.to(idx.dtype)
    codes = (idx | (torch.signbit(y).to(idx.dtype) << 3)).to(torch.uint8).reshape(r, k)
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    return packed.contiguous(), (se + 127).to(torch.uint8)


def _sub_seed(seed: int, tag: int, g: int) -> int:
    return (seed * 1_000_003 + tag * 104_729 + g) % (2 ** 62)


def _randn(shape, seed: int, device) -> torch.Tensor:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)


def draw_group_sizes(spec, G: int, seed: int) -> List[int]:
    """Valid rows per group for a size spec (numpy PCG64, platform independent)."""
    rng = np.random.default_rng(seed)
    kind = spec[0]
    if kind == "fixed":
        return [int(spec[1])] * G
    if kind == "uniform":  # inclusive bounds
        return [int(v) for v in rng.integers(spec[1], spec[2] + 1, size=G)]
    if kind == "dirichlet":
        p = rng.dirichlet([float(spec[1])] * G)
        return [int(v) for v in rng.multinomial(int(spec[2]), p)]
    if kind == "list":
        return [int(v) for v in spec[1]]
    raise ValueError(f"unknown size spec {spec!r}")


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclasses.dataclass
class Problem:
    """One grouped GEMM problem: e4m3 codes, fp32 UE8M0 scales and the row map."""

    name: str
    variant: str          # "contiguous" | "masked"
    G: int
    N: int
    K: int
    out_dtype: int
    sa_layout: int
    seed: int
    group_sizes: List[int]            # valid rows per group
    a: torch.Tensor                   # uint8 [M_sum, K] or [G, M_max, K]
    sa: torch.Tensor                  # fp32, layout per sa_layout
    ld_sa: int
    b: torch.Tensor                   # uint8 [G, N, K]
    sb: torch.Tensor                  # fp32 [G, N/128, K/128]
    grouped_layout: Optional[torch.Tensor] = None  # int32 [M_sum] (contiguous)
    masked_m: Optional[torch.Tensor] = None        # int32 [G] (masked)
    M_max: int = 0
    row_offsets: Optional[List[int]] = None        # contiguous: first row of each group
    pad_multiple: int = 128
    epilogue: str = ""    # "" (bf16/f16 D) or "silu_mul_quant" (E4M3 codes + scales of SiLU(gate)*up)
    scale_kind: str = "ue8m0"  # "ue8m0" / "fp32" (E4M3 with such scales) or "mxfp4"

    @property
    def KB(self) -> int:
        return self.K // 128

    @property
    def rows(self) -> int:
        """Rows of A as the kernel sees them (M_sum, or G*M_max)."""
        return self.a.shape[0] if self.variant == "contiguous" else self.G * self.M_max

    @property
    def valid_rows(self) -> int:
        return int(sum(self.group_sizes))

    @property
    def is_mx(self) -> bool:
        """MXFP4 operands: packed E2M1 [.., K/2] with E8M0 bytes [.., K/32]."""
        return self.scale_kind == "mxfp4"

    def flops(self) -> float:
        return 2.0 * self.valid_rows * self.N * self.K

    def algorithmic_bytes(self, out_bytes: int = 2) -> float:
        """A valid rows + B of groups with >=1 valid row + scales + D valid rows + row map."""
        used = sum(1 for m in self.group_sizes if m > 0)
        a = self.valid_rows * self.K
        b = used * self.N * self.K
        sa = self.valid_rows * self.KB * 4
        sb = used * (self.N // 128) * self.KB * 4
        if self.is_mx:   # half a byte per element, one scale byte per 32 along K (A and B rows)
            a, b = a // 2, b // 2
            sa = self.valid_rows * (self.K // 32)
            sb = used * self.N * (self.K // 32)
        d = self.valid_rows * self.N * out_bytes
        if self.epilogue == "silu_mul_quant":
            # N/2 code bytes and N/256 fp32 scales per row
            d = self.valid_rows * (self.N // 2 + (self.N // 256) * 4)
        rowmap = self.a.shape[0] * 4 if self.variant == "contiguous" else self.G * 4
        return float(a + b + sa + sb + d + rowmap)

    def regen_a_f32(self, g: int) -> torch.Tensor:
        """The pre-quantisation fp32 rows of group g (padding rows included)."""
        if self.variant == "contiguous":
            padded = self.row_offsets[g + 1] - self.row_offsets[g]
            return _randn((padded, self.K), _sub_seed(self.seed, 1, g), self.a.device)
        return _randn((self.M_max, self.K), _sub_seed(self.seed, 1, g), self.a.device)

    def regen_b_f32(self, g: int) -> torch.Tensor:
        return _randn((self.N, self.K), _sub_seed(self.seed, 2, g), self.b.device)

    def group_of_row(self, row: int):
        """(group, local row) of a flattened row index; group -1 for padding rows."""
        if self.variant == "masked":
            g, m = divmod(row, self.M_max)
            return (g, m) if m < self.group_sizes[g] else (-1, m)
        g = int(np.searchsorted(self.row_offsets, row, side="right")) - 1
        if g >= self.G:  # the ragged tail after the last group
            return (-1, row - self.row_offsets[-1])
        m = row - self.row_offsets[g]
        return (g, m) if m < self.group_sizes[g] else (-1, m)

    def sa_mk(self) -> torch.Tensor:
        """scale_a as [rows, K/128] regardless of the stored layout."""
        if self.sa_layout == SA_MK:
            return self.sa.reshape(-1, self.KB)
        if self.variant == "contiguous":
            return self.sa[:, : self.rows].t().contiguous()
        return self.sa[:, :, : self.M_max].permute(0, 2, 1).reshape(-1, self.KB).contiguous()

    def sa_mk_view(self) -> torch.Tensor:
        """scale_a as a logical [rows, K/128] (or [G, M_max, K/128]) tensor over the stored
        buffer: the buffer itself for SA_MK, a transposed view for SA_KM."""
        if self.sa_layout == SA_MK:
            return self.sa
        if self.variant == "contiguous":
            return self.sa[:, : self.rows].t()
        return self.sa[:, :, : self.M_max].transpose(1, 2)

    def to(self, device) -> "Problem":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return dataclasses.replace(self, a=mv(self.a), sa=mv(self.sa), b=mv(self.b), sb=mv(self.sb),
                                   grouped_layout=mv(self.grouped_layout), masked_m=mv(self.masked_m))


def make_problem(variant: str, G: int, N: int, K: int, group_sizes, *, out_dtype=OUT_BF16,
                 sa_layout=SA_MK, seed: int = 0, M_max: int = 0, pad_multiple: int = 128,
                 device="cpu", name: str = "custom", tail_rows: int = 0,
                 scale_kind: str = "ue8m0") -> Problem:
    """Build a problem from explicit group sizes.

    contiguous: group g owns round_up(group_sizes[g], pad_multiple) rows, the
    trailing ones marked -1; ``tail_rows`` extra -1 rows are appended at the
    end (a ragged M_sum).  masked: A is [G, M_max, K] and masked_m = group_sizes.
    Padding and masked rows hold random data too, so a kernel that wrongly
    computes or stores them is caught.  scale_kind "fp32" keeps each block's
    scale at amax / 448 instead of rounding it up to a power of two.
    """
    if scale_kind not in ("ue8m0", "fp32", "mxfp4"):
        raise ValueError(f"unknown scale_kind {scale_kind!r}")
    if scale_kind == "mxfp4":
        return _make_problem_mx(variant, G, N, K, group_sizes, out_dtype=out_dtype, seed=seed,
                                M_max=M_max, pad_multiple=pad_multiple, device=device, name=name,
                                tail_rows=tail_rows)
    pow2 = scale_kind == "ue8m0"
    sizes = [int(s) for s in group_sizes]
    if len(sizes) != G:
        raise ValueError("one size per group")
    KB = K // 128
    b_codes = torch.empty((G, N, K), dtype=torch.uint8, device=device)
    sb = torch.empty((G, N // 128, KB), dtype=torch.float32, device=device)
    for g in range(G):
        q, s = quantize_b_blocks(_randn((N, K), _sub_seed(seed, 2, g), device), pow2)
        b_codes[g] = q
        sb[g] = s
    if variant == "contiguous":
        offsets = [0]
        for m in sizes:
            offsets.append(offsets[-1] + _round_up(m, pad_multiple) if m > 0 else offsets[-1])
        m_sum = offsets[-1] + tail_rows
        a_codes = torch.empty((m_sum, K), dtype=torch.uint8, device=device)
        sa_mk = torch.empty((m_sum, KB), dtype=torch.float32, device=device)
        layout = torch.full((m_sum,), -1, dtype=torch.int32, device=device)
        for g in range(G):
            lo, hi = offsets[g], offsets[g + 1]
            if hi > lo:
                q, s = quantize_a_blocks(_randn((hi - lo, K), _sub_seed(seed, 1, g), device), pow2)
                a_codes[lo:hi] = q
                sa_mk[lo:hi] = s
                layout[lo:lo + sizes[g]] = g
        if tail_rows:
            q, s = quantize_a_blocks(_randn((tail_rows, K), _sub_seed(seed, 3, 0), device), pow2)
            a_codes[offsets[-1]:] = q
            sa_mk[offsets[-1]:] = s
        if sa_layout == SA_KM:
            ld = _round_up(m_sum, 4)
            sa = torch.zeros((KB, ld), dtype=torch.float32, device=device)
            sa[:, :m_sum] = sa_mk.t()
        else:
            ld, sa = KB, sa_mk
        return Problem(name=name, variant=variant, G=G, N=N, K=K, out_dtype=out_dtype,
                       sa_layout=sa_layout, seed=seed, group_sizes=sizes, a=a_codes, sa=sa,
                       ld_sa=ld, b=b_codes, sb=sb, grouped_layout=layout, row_offsets=offsets,
                       pad_multiple=pad_multiple, scale_kind=scale_kind)
    if variant == "masked":
        if M_max <= 0 or max(sizes) > M_max:
            raise ValueError("masked: need 0 < max(masked_m) <= M_max")
        a_codes = torch.empty((G, M_max, K), dtype=torch.uint8, device=device)
        sa_mk = torch.empty((G, M_max, KB), dtype=torch.float32, device=device)
        for g in range(G):
            q, s = quantize_a_blocks(_randn((M_max, K), _sub_seed(seed, 1, g), device), pow2)
            a_codes[g] = q
            sa_mk[g] = s
        if sa_layout == SA_KM:
            ld = _round_up(M_max, 4)
            sa = torch.zeros((G, KB, ld), dtype=torch.float32, device=device)
            sa[:, :, :M_max] = sa_mk.permute(0, 2, 1)
        else:
            ld, sa = KB, sa_mk
        mm = torch.tensor(sizes, dtype=torch.int32, device=device)
        return Problem(name=name, variant=variant, G=G, N=N, K=K, out_dtype=out_dtype,
                       sa_layout=sa_layout, seed=seed, group_sizes=sizes, a=a_codes, sa=sa,
                       ld_sa=ld, b=b_codes, sb=sb, masked_m=mm, M_max=M_max, scale_kind=scale_kind)
    raise ValueError(f"unknown variant {variant!r}")


def _make_problem_mx(variant, G, N, K, group_sizes, *, out_dtype, seed, M_max, pad_multiple,
                     device, name, tail_rows) -> Problem:
    """make_problem for MXFP4 operands (same data draws, quantize_mxfp4)."""
    sizes = [int(s) for s in group_sizes]
    if len(sizes) != G:
        raise ValueError("one size per group")
    if K % 256:
        raise ValueError("MXFP4 workloads need K % 256 == 0")
    b = torch.empty((G, N, K // 2), dtype=torch.uint8, device=device)
    sb = torch.empty((G, N, K // 32), dtype=torch.uint8, device=device)
    for g in range(G):
        b[g], sb[g] = quantize_mxfp4(_randn((N, K), _sub_seed(seed, 2, g), device))
    common = dict(name=name, variant=variant, G=G, N=N, K=K, out_dtype=out_dtype,
                  sa_layout=SA_MK, seed=seed, group_sizes=sizes, ld_sa=K // 32, b=b, sb=sb,
                  scale_kind="mxfp4")
    if variant == "contiguous":
        offsets = [0]
        for m in sizes:
            offsets.append(offsets[-1] + _round_up(m, pad_multiple) if m > 0 else offsets[-1])
        m_sum = offsets[-1] + tail_rows
        a = torch.empty((m_sum, K // 2), dtype=torch.uint8, device=device)
        sa = torch.empty((m_sum, K // 32), dtype=torch.uint8, device=device)
        layout = torch.full((m_sum,), -1, dtype=torch.int32, device=device)
        for g in range(G):
            lo, hi = offsets[g], offsets[g + 1]
            if hi > lo:
                a[lo:hi], sa[lo:hi] = quantize_mxfp4(_randn((hi - lo, K), _sub_seed(seed, 1, g),
                                                            device))
                layout[lo:lo + sizes[g]] = g
        if tail_rows:
            a[offsets[-1]:], sa[offsets[-1]:] = quantize_mxfp4(
                _randn((tail_rows, K), _sub_seed(seed, 3, 0), device))
        return Problem(a=a, sa=sa, grouped_layout=layout, row_offsets=offsets,
                       pad_multiple=pad_multiple, **common)
    if variant == "masked":
        if M_max <= 0 or max(sizes) > M_max:
            raise ValueError("masked: need 0 < max(masked_m) <= M_max")
        a = torch.empty((G, M_max, K // 2), dtype=torch.uint8, device=device)
        sa = torch.empty((G, M_max, K // 32), dtype=torch.uint8, device=device)
        for g in range(G):
            a[g], sa[g] = quantize_mxfp4(_randn((M_max, K), _sub_seed(seed, 1, g), device))
        mm = torch.tensor(sizes, dtype=torch.int32, device=device)
        return Problem(a=a, sa=sa, masked_m=mm, M_max=M_max, **common)
    raise ValueError(f"unknown variant {variant!r}")


def make_config(name: str, device="cpu") -> Problem:
    """One of the named workloads of CONFIGS."""
    c = CONFIGS[name]
    sizes = draw_group_sizes(c["sizes"], c["G"], c["seed"])
    p = make_problem(c["variant"], c["G"], c["N"], c["K"], sizes, out_dtype=c["out"],
                     sa_layout=c["sa_layout"], seed=c["seed"], M_max=c.get("M_max", 0),
                     device=device, name=name, scale_kind=c.get("scale_kind", "ue8m0"))
    p.epilogue = c.get("epilogue", "")
    return p


def sample_rows(p: Problem, per_group: int = 32, seed: int = 0):
    """Seeded row sample for checking a large problem row by row.

    valid_rows, per group: the first and last valid rows, ``per_group`` uniform
    random valid rows, and one random valid row of every 128-row tile of the
    group (the kernels' row tiles: a contiguous expert starts on a tile
    boundary, a masked group's tiles start at its row 0), so that every tile
    the kernel computes is compared.  untouched_rows: every row that must keep
    its prior contents (padding rows, rows past masked_m, the ragged tail).
    Indices are flattened rows of A (contiguous: global row; masked: g*M_max+m).
    """
    rng = np.random.default_rng(10_007 + seed)
    valid, untouched = [], []
    for g, m in enumerate(p.group_sizes):
        base = p.row_offsets[g] if p.variant == "contiguous" else g * p.M_max
        span = (p.row_offsets[g + 1] - p.row_offsets[g]) if p.variant == "contiguous" else p.M_max
        if m > 0:
            picks = {0, m - 1}
            picks.update(int(v) for v in rng.integers(0, m, size=min(per_group, m)))
            for t0 in range(0, m, 128):
                picks.add(t0 + int(rng.integers(0, min(128, m - t0))))
            valid.extend(base + v for v in sorted(picks))
        untouched.extend(range(base + m, base + span))
    if p.variant == "contiguous":
        untouched.extend(range(p.row_offsets[-1], p.rows))  # ragged tail after the last group
    return (np.array(sorted(set(valid)), dtype=np.int64),
            np.array(sorted(set(untouched)), dtype=np.int64))


__all__ = ["CONFIGS", "Problem", "make_problem", "make_config", "quantize_a_blocks", "quantize_mxfp4",
           "quantize_b_blocks", "ceil_to_ue8m0_f32", "draw_group_sizes", "sample_rows",
           "SA_MK", "SA_KM", "OUT_BF16", "OUT_F16"]
