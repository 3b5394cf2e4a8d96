/*
 * CPU oracle for the grouped FP8 (e4m3) block-scaled GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only tests/, __graft_entry__.smoke() and the cpu_baseline /
 * reference leg of bench.py use it.  It shares no code, header, table or
 * constant with the CUDA library under fp8_block_scaled_gb300/.
 *
 * Everything is written from the definitions, in fp64, in the plainest
 * order: no blocking, no fusion, no reordering beyond what the definition
 * states.  Each function cites the passage it follows:
 *
 *   [P1] "Adds Grouped and Batched GEMM kernels with blockscaling matching
 *        DeepGEMM API" (FlyDSL PR #433):
 *          - Summary: grouped (contiguous, grouped_layout with -1 for padding)
 *            and masked (masked_m) variants, (1,128) x (128,128) block-scale
 *            granularity, transposed [scale_k, M] activation-scale layout.
 *          - DeepGEMM conformance details: calc_diff tolerance metric,
 *            ceil_to_ue8m0 scale rounding, reference from pre-quantisation
 *            fp32, E8M0 scales applied by the matrix instruction.
 *          - Notes for reviewers: the dequant-then-matmul reference style.
 *   [OFP8] the OCP 8-bit floating point format E4M3 ("FN": bias 7, no
 *          infinities, S.1111.111 is NaN, max normal 448).
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_SA_MK 0 /* scale_a stored [rows, K/128]            */
#define ORACLE_SA_KM 1 /* scale_a stored transposed [K/128, ld_sa] */

int fp8bs_oracle_abi_version(void) { return 1; }

int fp8bs_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* [OFP8] E4M3 decode: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 holds subnormals m/8 * 2^-6.  S.1111.111 is NaN; there is
 * no infinity, so exponent field 15 with m < 7 is an ordinary normal. */
double fp8bs_oracle_e4m3_to_double(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* [OFP8] fp64 -> E4M3 with round-to-nearest, ties to an even mantissa, and
 * saturation of finite magnitudes above 448 to 448 (the pages fix no
 * overflow rule; with ceil_to_ue8m0 scales |x/s| <= 448 so it never fires).
 * Written as a search over the 127 non-negative finite codes so that it is
 * obviously the nearest representable value.  NaN maps to 0x7F. */
uint8_t fp8bs_oracle_double_to_e4m3(double x) {
    double ax;
    int best = 0, c;
    double best_err;
    if (isnan(x)) return 0x7F;
    ax = fabs(x);
    if (ax > 448.0) ax = 448.0;
    best_err = INFINITY;
    for (c = 0; c <= 0x7E; ++c) {
        double v = fp8bs_oracle_e4m3_to_double((uint8_t)c);
        double err = fabs(v - ax);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best_err = err;
            best = c;
        }
    }
    if (signbit(x)) best |= 0x80;
    return (uint8_t)best;
}

/* [P1 DeepGEMM conformance] ceil_to_ue8m0: the smallest power of two that is
 * >= t (t > 0, finite).  frexp gives t = f * 2^E with f in [0.5, 1); t is a
 * power of two exactly when f == 0.5. */
double fp8bs_oracle_ceil_to_ue8m0(double t) {
    int E;
    double f;
    if (!(t > 0.0) || isinf(t)) return NAN;
    f = frexp(t, &E);
    if (f == 0.5) return t;
    return ldexp(1.0, E);
}

/* Round an fp64 value to a binary format with p significant bits, minimum
 * normal exponent emin and largest finite value maxval, round-to-nearest-even
 * (IEEE 754 default).  Overflow beyond the rounding boundary gives +-inf. */
static double round_to_format(double x, int p, int emin, int emax) {
    int E;
    int lead;
    double quantum, q, r, y, maxval, limit;
    if (x == 0.0 || isnan(x) || isinf(x)) return x;
    frexp(fabs(x), &E);   /* |x| = f * 2^E, leading bit at 2^(E-1) */
    lead = E - 1;
    if (lead < emin) lead = emin; /* subnormal: fixed quantum */
    quantum = ldexp(1.0, lead - (p - 1));
    q = x / quantum;              /* exact: power-of-two scaling */
    r = nearbyint(q);             /* default mode: nearest, ties to even */
    y = r * quantum;
    maxval = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    limit = ldexp(2.0 - ldexp(1.0, -p), emax); /* max + half ulp */
    if (fabs(x) >= limit) return signbit(x) ? -INFINITY : INFINITY;
    if (fabs(y) > maxval) y = signbit(x) ? -maxval : maxval;
    return y;
}

/* Encode a value that is exactly representable in a format with 1 sign bit,
 * `ebits` exponent bits (bias 2^(ebits-1)-1) and `mbits` mantissa bits. */
static uint16_t encode_exact(double y, int ebits, int mbits) {
    int bias = (1 << (ebits - 1)) - 1;
    uint16_t sign = signbit(y) ? 1 : 0;
    uint16_t expf, mant;
    double ay = fabs(y);
    if (isnan(y)) return (uint16_t)(((1u << ebits) - 1) << mbits | (1u << (mbits - 1)));
    if (isinf(y)) return (uint16_t)((sign << (ebits + mbits)) | (((1u << ebits) - 1) << mbits));
    if (ay == 0.0) return (uint16_t)(sign << (ebits + mbits));
    {
        int E;
        double f = frexp(ay, &E); /* ay = f * 2^E, f in [0.5,1) */
        int e = E - 1;             /* ay = (2f) * 2^e, 2f in [1,2) */
        if (e < 1 - bias) {        /* subnormal */
            expf = 0;
            mant = (uint16_t)ldexp(ay, (bias - 1) + mbits);
        } else {
            expf = (uint16_t)(e + bias);
            mant = (uint16_t)ldexp(2.0 * f - 1.0, mbits);
        }
    }
    return (uint16_t)((sign << (ebits + mbits)) | (expf << mbits) | mant);
}

/* fp64 -> bf16 bits (8 exponent bits, 7 mantissa bits), RNE. */
uint16_t fp8bs_oracle_round_bf16(double x) {
    return encode_exact(round_to_format(x, 8, -126, 127), 8, 7);
}

/* fp64 -> IEEE binary16 bits (5 exponent bits, 10 mantissa bits), RNE. */
uint16_t fp8bs_oracle_round_f16(double x) {
    return encode_exact(round_to_format(x, 11, -14, 15), 5, 10);
}

void fp8bs_oracle_round_array(const double* x, int64_t count, int out_dtype, uint16_t* bits) {
    int64_t i;
    for (i = 0; i < count; ++i)
        bits[i] = out_dtype == 0 ? fp8bs_oracle_round_bf16(x[i]) : fp8bs_oracle_round_f16(x[i]);
}

/* Read scale_a for flattened A row `row` (its local row index within the
 * group is `mloc`, its group is `g`) and K-block kb, in either layout.
 *   MK: sa[row * KB + kb]           (contiguous: [M_sum, KB]; masked: [G*M_max, KB])
 *   KM: sa[g * g_stride + kb * ld_sa + mloc]  (contiguous: g_stride = 0,
 *       mloc = row; masked: [G, KB, ld_sa], g_stride = KB * ld_sa) */
static double read_sa(const float* sa, int sa_layout, int64_t ld_sa, int64_t KB, int64_t row,
                      int64_t g, int64_t mloc, int masked, int64_t kb) {
    if (sa_layout == ORACLE_SA_MK) return (double)sa[row * KB + kb];
    if (masked) return (double)sa[g * KB * ld_sa + kb * ld_sa + mloc];
    return (double)sa[kb * ld_sa + row];
}

/* The 256 E4M3 values, index = byte code, each from the decode above. */
static void decode_table(double* dec) {
    int c;
    for (c = 0; c < 256; ++c) dec[c] = fp8bs_oracle_e4m3_to_double((uint8_t)c);
}

/* One output row of the grouped GEMM, straight from the definition
 *   acc[n] = sum_kb sa[r,kb] * sb[g, n/128, kb]
 *                   * sum_{k in block kb} e4m3(A[r,k]) * e4m3(B[g,n,k])
 * ([P1 Summary]: (1,128) activation and (128,128) weight granularity),
 * everything in fp64. */
static void one_row(const uint8_t* a, const float* sa, int sa_layout, int64_t ld_sa,
                    const uint8_t* b, const float* sb, int64_t row, int64_t g, int64_t mloc,
                    int masked, int64_t n_dim, int64_t k_dim, const double* dec,
                    double* acc) {
    int64_t KB = k_dim / 128, NB = n_dim / 128;
    int64_t n, kb, k;
    for (n = 0; n < n_dim; ++n) {
        double total = 0.0;
        for (kb = 0; kb < KB; ++kb) {
            double dot = 0.0;
            double s_a = read_sa(sa, sa_layout, ld_sa, KB, row, g, mloc, masked, kb);
            double s_b = (double)sb[(g * NB + n / 128) * KB + kb];
            for (k = kb * 128; k < kb * 128 + 128; ++k) {
                double x = dec[a[row * k_dim + k]];
                double y = dec[b[(g * n_dim + n) * k_dim + k]];
                dot += x * y;
            }
            total += (s_a * s_b) * dot;
        }
        acc[n] = total;
    }
}

/* Contiguous variant [P1 Summary]: A [M_sum, K], grouped_layout[r] is the
 * expert of row r, -1 marks a padding row that produces no output.
 * Computes the rows listed in rows[0..nrows); acc is [nrows, N].
 * valid[i] is set to 1 for a computed row, 0 for a padding row (its acc row
 * is left as NaN).  Returns 0, or -1 on an out-of-range argument. */
int fp8bs_oracle_contiguous(const uint8_t* a, const float* sa, int sa_layout, int64_t ld_sa,
                            const uint8_t* b, const float* sb, const int32_t* grouped_layout,
                            int64_t m_sum, int64_t n_dim, int64_t k_dim, int64_t num_groups,
                            const int64_t* rows, int64_t nrows, double* acc, uint8_t* valid) {
    int64_t i;
    int bad = 0;
    double dec[256];
    if (k_dim % 128 || n_dim % 128) return -1;
    decode_table(dec);
    for (i = 0; i < nrows; ++i) {
        int64_t r = rows[i];
        if (r < 0 || r >= m_sum) bad = 1;
        else if (grouped_layout[r] >= num_groups || grouped_layout[r] < -1) bad = 1;
    }
    if (bad) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < nrows; ++i) {
        int64_t r = rows[i];
        int64_t g = grouped_layout[r];
        int64_t n;
        if (g < 0) {
            valid[i] = 0;
            for (n = 0; n < n_dim; ++n) acc[i * n_dim + n] = NAN;
            continue;
        }
        valid[i] = 1;
        one_row(a, sa, sa_layout, ld_sa, b, sb, r, g, r, 0, n_dim, k_dim, dec, acc + i * n_dim);
    }
    return 0;
}

/* Masked variant [P1 Summary]: A [G, M_max, K]; only the first masked_m[g]
 * rows of group g are computed.  rows[] holds flattened indices g*M_max + m. */
int fp8bs_oracle_masked(const uint8_t* a, const float* sa, int sa_layout, int64_t ld_sa,
                        const uint8_t* b, const float* sb, const int32_t* masked_m,
                        int64_t num_groups, int64_t m_max, int64_t n_dim, int64_t k_dim,
                        const int64_t* rows, int64_t nrows, double* acc, uint8_t* valid) {
    int64_t i;
    int bad = 0;
    double dec[256];
    if (k_dim % 128 || n_dim % 128) return -1;
    decode_table(dec);
    for (i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= num_groups * m_max) bad = 1;
    for (i = 0; i < num_groups; ++i)
        if (masked_m[i] < 0 || masked_m[i] > m_max) bad = 1;
    if (bad) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < nrows; ++i) {
        int64_t f = rows[i];
        int64_t g = f / m_max, m = f % m_max;
        int64_t n;
        if (m >= masked_m[g]) {
            valid[i] = 0;
            for (n = 0; n < n_dim; ++n) acc[i * n_dim + n] = NAN;
            continue;
        }
        valid[i] = 1;
        one_row(a, sa, sa_layout, ld_sa, b, sb, f, g, m, 1, n_dim, k_dim, dec, acc + i * n_dim);
    }
    return 0;
}

/* [P1 DeepGEMM conformance] calc_diff, the cosine-similarity-style normalised
 * error: 1 - 2*sum(x*y) / (sum(x^2) + sum(y^2)), in fp64.  Defined as 0 when
 * both vectors are zero. */
double fp8bs_oracle_calc_diff(const double* x, const double* y, int64_t count) {
    double sxy = 0.0, sxx = 0.0, syy = 0.0;
    int64_t i;
    for (i = 0; i < count; ++i) {
        sxy += x[i] * y[i];
        sxx += x[i] * x[i];
        syy += y[i] * y[i];
    }
    if (sxx + syy == 0.0) return 0.0;
    return 1.0 - 2.0 * sxy / (sxx + syy);
}

/* Exactness witness for one 128-element block product: every E4M3 value is an
 * integer multiple of 2^-9 (the smallest subnormal), so the block sum is an
 * integer multiple of 2^-18 whose magnitude stays below 128 * (448*2^9)^2
 * < 2^43.  Returns the block sum computed in int64 units of 2^-18, scaled
 * back exactly; the pins compare it with the fp64 sum. */
double fp8bs_oracle_block_dot_exact(const uint8_t* x, const uint8_t* y) {
    int64_t total = 0;
    int k;
    for (k = 0; k < 128; ++k) {
        double vx = fp8bs_oracle_e4m3_to_double(x[k]);
        double vy = fp8bs_oracle_e4m3_to_double(y[k]);
        int64_t ix = (int64_t)ldexp(vx, 9);
        int64_t iy = (int64_t)ldexp(vy, 9);
        total += ix * iy;
    }
    return ldexp((double)total, -18);
}

/* ------------------------------------------------------------------------
 * Fused MoE gate/up epilogue: SiLU(gate) * up, requantised for the down
 * projection.
 *
 * [P3] "flydsl mxfp4 a4w4 MoE: bring gemm1/gemm2 to parity with the HIP
 *      backend", section gemm1: the first MoE GEMM ends in silu_mul, i.e. the
 *      SiLU of the gate half of its output times the up half.
 * [P1] Summary and DeepGEMM conformance details: the down projection consumes
 *      E4M3 activations with (1,128) UE8M0 ceil scales, the quantiser of the
 *      inputs (amax / 448, ceil to a power of two, round to nearest even).
 *
 * gate, up: the fp64 accumulators of the two halves, rows x I, row stride ld.
 * For every row and column j < I:
 *     h = gate / (1 + exp(-gate)) * up                            (fp64)
 * and per 128-column block of a row:
 *     amax = max |h| (at least 1e-4, the reading for an all-zero block),
 *     t = fl32(fl32(amax) / 448), s = ceil_to_ue8m0(t),
 *     q = e4m3_rne(fl32(h) / s)
 * The scale exponent and the codes are decided in fp32 (the kernel's
 * precision; the pages fix none).  Outputs, all rows x I unless noted:
 *     h       the exact (fp64) activation;
 *     q       E4M3 codes;
 *     s       [rows, I/128] scales;
 *     margin  relative distance of fl32(h)/s to the nearest E4M3 rounding
 *             boundary (the midpoint between two neighbouring values);
 *     tmargin [rows, I/128] relative distance of amax/448 (fp64) to the
 *             nearest power of two.
 * Where a margin is tiny, an accumulator that differs from the exact one in
 * its last fp32 bits may round to the other neighbour (several results are
 * correct); everywhere else the code and the scale are unique.
 * ------------------------------------------------------------------------ */
static double e4m3_boundary_margin(double x) {
    /* boundaries between neighbouring non-negative E4M3 values, and the
     * relative distance of |x| to the nearest of them */
    double ax = fabs(x), best = INFINITY, prev, cur, mid, d;
    int c;
    prev = fp8bs_oracle_e4m3_to_double(0);
    for (c = 1; c <= 0x7E; ++c) {
        cur = fp8bs_oracle_e4m3_to_double((uint8_t)c);
        mid = 0.5 * (prev + cur);
        d = fabs(ax - mid);
        if (d < best) best = d;
        prev = cur;
    }
    return best / (ax > ldexp(1.0, -9) ? ax : ldexp(1.0, -9));
}

int fp8bs_oracle_silu_mul_quant(const double* gate, const double* up, int64_t rows, int64_t ld,
                                int64_t I, double* h, uint8_t* q, float* s, double* margin,
                                double* tmargin) {
    int64_t r;
    if (rows < 0 || I <= 0 || I % 128 != 0 || ld < I) return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < rows; ++r) {
        int64_t jb, j;
        for (jb = 0; jb < I / 128; ++jb) {
            double amax = 0.0, t64, f;
            float t, sc;
            int E;
            for (j = jb * 128; j < jb * 128 + 128; ++j) {
                const double g = gate[r * ld + j];
                const double v = g / (1.0 + exp(-g)) * up[r * ld + j];
                h[r * I + j] = v;
                if (fabs(v) > amax) amax = fabs(v);
            }
            if (amax < 1e-4) amax = 1e-4;
            t = (float)amax / 448.0f;
            sc = (float)fp8bs_oracle_ceil_to_ue8m0((double)t);
            s[r * (I / 128) + jb] = sc;
            t64 = amax / 448.0;
            f = frexp(t64, &E); /* t64 = f * 2^E, f in [0.5, 1) */
            tmargin[r * (I / 128) + jb] = fmin(2.0 * f - 1.0, (1.0 - f) / f);
            for (j = jb * 128; j < jb * 128 + 128; ++j) {
                const float x = (float)h[r * I + j] / sc; /* exact: sc is a power of two */
                q[r * I + j] = fp8bs_oracle_double_to_e4m3((double)x);
                margin[r * I + j] = e4m3_boundary_margin((double)x);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * MXFP4 (a4w4) grouped GEMM.
 *
 * [P3] "flydsl mxfp4 a4w4 MoE: bring gemm1/gemm2 to parity with the HIP
 *      backend", Summary: the MoE GEMMs with both operands in MXFP4.
 * [OMX] the OCP Microscaling (MX) formats: E2M1 elements -- a sign bit, two
 *      exponent bits with bias 1 and one mantissa bit, magnitudes 0, 0.5, 1,
 *      1.5, 2, 3, 4, 6, no infinity or NaN -- in blocks of 32 consecutive
 *      elements along K that share one E8M0 scale 2^(e - 127) (e = 255 is NaN).
 *
 * Storage: two elements per byte, element 2i in the low nibble of byte i;
 * scales one byte each, sa [rows, K/32] (masked: [G, M_max, K/32]) and
 * sb [G, N, K/32].  For every computed row r of group g and column n:
 *     acc = sum_j 2^(sa[r,j]-127) * 2^(sb[g,n,j]-127)
 *                 * sum_{k in block j} e2m1(A[r,k]) * e2m1(B[g,n,k])      (fp64)
 * Every block sum is a multiple of 1/4 below 32 * 36 and the scales are
 * powers of two, so acc is exact while the scale exponents span less than
 * about 40 binades.
 * ------------------------------------------------------------------------ */
double fp8bs_oracle_e2m1_to_double(uint8_t code) {
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

double fp8bs_oracle_e8m0_to_double(uint8_t e) {
    if (e == 0xFF) return NAN;
    return ldexp(1.0, (int)e - 127);
}

static double e2m1_at(const uint8_t* packed, int64_t row_bytes, int64_t row, int64_t k) {
    const uint8_t byte = packed[row * row_bytes + k / 2];
    return fp8bs_oracle_e2m1_to_double((uint8_t)((k & 1) ? (byte >> 4) : (byte & 0xF)));
}

static void mx_row(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                   int64_t arow, int64_t g, int64_t n_dim, int64_t k_dim, double* acc) {
    const int64_t nblk = k_dim / 32;
    int64_t n, j, k;
    for (n = 0; n < n_dim; ++n) {
        const int64_t brow = g * n_dim + n;
        double total = 0.0;
        for (j = 0; j < nblk; ++j) {
            double dot = 0.0;
            for (k = j * 32; k < j * 32 + 32; ++k)
                dot += e2m1_at(a, k_dim / 2, arow, k) * e2m1_at(b, k_dim / 2, brow, k);
            total += fp8bs_oracle_e8m0_to_double(sa[arow * nblk + j]) *
                     fp8bs_oracle_e8m0_to_double(sb[brow * nblk + j]) * dot;
        }
        acc[n] = total;
    }
}

int fp8bs_oracle_mxfp4_contiguous(const uint8_t* a, const uint8_t* sa, const uint8_t* b,
                                  const uint8_t* sb, const int32_t* grouped_layout,
                                  int64_t m_sum, int64_t n_dim, int64_t k_dim,
                                  int64_t num_groups, const int64_t* rows, int64_t nrows,
                                  double* acc, uint8_t* valid) {
    int64_t i;
    int bad = 0;
    if (k_dim % 32 || n_dim <= 0) return -1;
    for (i = 0; i < nrows; ++i) {
        int64_t r = rows[i];
        if (r < 0 || r >= m_sum) bad = 1;
        else if (grouped_layout[r] >= num_groups || grouped_layout[r] < -1) bad = 1;
    }
    if (bad) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < nrows; ++i) {
        int64_t r = rows[i];
        int64_t g = grouped_layout[r];
        int64_t n;
        if (g < 0) {
            valid[i] = 0;
            for (n = 0; n < n_dim; ++n) acc[i * n_dim + n] = NAN;
            continue;
        }
        valid[i] = 1;
        mx_row(a, sa, b, sb, r, g, n_dim, k_dim, acc + i * n_dim);
    }
    return 0;
}

int fp8bs_oracle_mxfp4_masked(const uint8_t* a, const uint8_t* sa, const uint8_t* b,
                              const uint8_t* sb, const int32_t* masked_m, int64_t num_groups,
                              int64_t m_max, int64_t n_dim, int64_t k_dim, const int64_t* rows,
                              int64_t nrows, double* acc, uint8_t* valid) {
    int64_t i;
    int bad = 0;
    if (k_dim % 32 || n_dim <= 0) return -1;
    for (i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= num_groups * m_max) bad = 1;
    for (i = 0; i < num_groups; ++i)
        if (masked_m[i] < 0 || masked_m[i] > m_max) bad = 1;
    if (bad) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < nrows; ++i) {
        int64_t f = rows[i];
        int64_t g = f / m_max, m = f % m_max;
        int64_t n;
        if (m >= masked_m[g]) {
            valid[i] = 0;
            for (n = 0; n < n_dim; ++n) acc[i * n_dim + n] = NAN;
            continue;
        }
        valid[i] = 1;
        mx_row(a, sa, b, sb, f, g, n_dim, k_dim, acc + i * n_dim);
    }
    return 0;
}
