// Scale pre-pass of the E4M3 CTA-pair kernel.
//
// The block-scaled MMA ("Adds Grouped and Batched GEMM kernels with blockscaling
// matching DeepGEMM API", section DeepGEMM conformance details: UE8M0 scales
// applied by the matrix instruction) reads its scales from tensor memory as
// UE8M0 bytes, copied there per pipeline step by tcgen05.cp from shared memory.
// This kernel turns the fp32 scales of a whole call into exactly those shared-
// memory images once, ahead of the GEMM, so that the GEMM only copies 1.5 KB per
// step and CTA into shared memory instead of gathering and converting the fp32
// values in its pipeline.  The library runs it for row-major activation scales,
// whose in-kernel fetch is a gather of one 8-byte pair per row and step:
//
//   packed A: [scale tile t][step ks][128 words], 512 bytes per (t, ks): the
//             word at position 4 l + q is row 32 q + l of 128-row tile t (the
//             32x128b.warpx4 source order), byte j the UE8M0 code of K block
//             2 ks + j % 2 of that row (zero past K and past the rows).  Tile t
//             is the global 128-row tile of the contiguous layout, or tile
//             t % tiles_per_group of group t / tiles_per_group when masked.
//   packed B: [g * N/128 + nb][step ks][128 words]: the same word, byte j the
//             code of weight block (g, nb, 2 ks + j % 2), repeated 128 times (the
//             weight scales of a 128-column chunk are replicated over its rows).
//
// The activation scales of every row the GEMM stores (contiguous: the row's
// group is its tile's, the group of the tile's first row, and not -1; masked:
// row < masked_m[g]) are checked to be UE8M0 values and FP8BS_DEVERR_BAD_SCALE
// is raised otherwise; the GEMM checks the weight scales of the units it runs.
#pragma once

#include "grouped_gemm.cuh"

namespace fp8bs {

struct ScalePackParams {
    const float* sa;
    const float* sb;
    const int32_t* row_info;   // contiguous: grouped_layout [rows]; masked: masked_m [G]
    uint32_t* packed_a;        // 16-byte aligned
    uint32_t* packed_b;        // 16-byte aligned
    uint32_t* err;
    int64_t rows;              // contiguous: m_sum; masked: m_max
    int64_t sa_g_stride, sa_kb_stride, sa_row_stride;
    uint32_t a_vecs;           // 16-byte vectors of packed A: tiles * steps * 32
    uint32_t b_vecs;           // 16-byte vectors of packed B: G * N/128 * steps * 32
    int kb_count, steps, tiles_per_group, masked;
};

// the UE8M0 codes of K blocks 2 ks and 2 ks + 1 as one image word: bytes c0, c1, c0, c1
__device__ __forceinline__ uint32_t image_word(uint32_t f0, uint32_t f1) {
    return (((f0 >> 23) & 0xFFu) | (((f1 >> 23) & 0xFFu) << 8)) * 0x00010001u;
}

// A warp writes one 512-byte image at a time, lane l one 16-byte vector of it: four
// words of a (tile, step) image, rows l, 32 + l, 64 + l and 96 + l of the tile
// (words 4 l .. 4 l + 3), or four copies of a weight-scale word.  Consecutive images
// go to consecutive blocks, so that the activation images (gathers of scattered
// rows, the costly part) are spread over every block and SM rather than left to
// the first few.
__global__ void __launch_bounds__(256) scale_pack_kernel(const ScalePackParams p) {
    // the scales may be written by the grid this launch follows, and the workspace
    // may still be read by it (programmatic dependent launch)
    grid_dependency_wait();
    grid_launch_dependents();
    const uint32_t images = (p.a_vecs + p.b_vecs) >> 5;
    const uint32_t warps = gridDim.x * (blockDim.x >> 5);
    const uint32_t steps = static_cast<uint32_t>(p.steps);
    const uint32_t lane = threadIdx.x & 31u;
    bool bad = false;
    for (uint32_t img = (threadIdx.x >> 5) * gridDim.x + blockIdx.x; img < images; img += warps) {
        const uint32_t v = img * 32u + lane;
        if (v < p.a_vecs) {
            const uint32_t tk = v >> 5;                    // (tile, step)
            const uint32_t t = tk / steps;
            const int ks = static_cast<int>(tk - t * steps);
            const int l = static_cast<int>(v & 31u);
            int64_t m0, sa_goff = 0;
            int mm = 0, tg = 0;
            if (p.masked) {
                const uint32_t g = t / static_cast<uint32_t>(p.tiles_per_group);
                m0 = static_cast<int64_t>(t - g * p.tiles_per_group) * kBM;
                mm = __ldg(p.row_info + g);
                mm = mm < 0 ? 0 : (mm > p.rows ? static_cast<int>(p.rows) : mm);
                // no unit reads a tile past masked_m[g] (the second tile of a pair
                // whose first one holds rows is read, by its idle half): not written
                if (!(m0 < mm || (m0 >= kBM && m0 - kBM < mm))) continue;
                sa_goff = static_cast<int64_t>(g) * p.sa_g_stride;
            } else {
                m0 = static_cast<int64_t>(t) * kBM;
                tg = __ldg(p.row_info + m0);               // the tile's group
            }
            uint32_t f[4][2];
            bool stored[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t m = m0 + q * 32 + l;
                const bool in = m < p.rows;
                stored[q] = p.masked ? m < mm : in && tg >= 0 && __ldg(p.row_info + m) == tg;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int kb = 2 * ks + j;
                    f[q][j] = in && kb < p.kb_count
                                  ? __float_as_uint(__ldg(p.sa + sa_goff + kb * p.sa_kb_stride +
                                                          m * p.sa_row_stride))
                                  : 0u;
                }
            }
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    bad |= stored[q] && 2 * ks + j < p.kb_count && !ue8m0_scale_ok(f[q][j]);
                w[q] = image_word(f[q][0], f[q][1]);
            }
            st_global_v4(p.packed_a + static_cast<int64_t>(v) * 4, w[0], w[1], w[2], w[3]);
        } else {
            const uint32_t vb = v - p.a_vecs;
            const uint32_t ck = vb >> 5;                   // (g * N/128 + nb, step)
            const uint32_t c = ck / steps;
            const int ks = static_cast<int>(ck - c * steps);
            const float* src = p.sb + static_cast<int64_t>(c) * p.kb_count + 2 * ks;
            const uint32_t f0 = __float_as_uint(__ldg(src));
            const uint32_t f1 = 2 * ks + 1 < p.kb_count ? __float_as_uint(__ldg(src + 1)) : 0u;
            const uint32_t w = image_word(f0, f1);
            st_global_v4(p.packed_b + static_cast<int64_t>(vb) * 4, w, w, w, w);
        }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) raise_error(p.err, kErrBadScale);
}

}  // namespace fp8bs
