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
    uint32_t* packed_a;
    uint32_t* packed_b;
    uint32_t* err;
    int64_t rows;              // contiguous: m_sum; masked: m_max
    int64_t sa_g_stride, sa_kb_stride, sa_row_stride;
    int64_t a_words;           // tiles * steps * 128
    int64_t b_words;           // G * N/128 * steps * 128
    int kb_count, steps, tiles_per_group, masked;
};

__device__ __forceinline__ uint32_t ue8m0_code(uint32_t fbits) { return (fbits >> 23) & 0xFFu; }

__global__ void __launch_bounds__(256) scale_pack_kernel(const ScalePackParams p) {
    // the scales may be written by the grid this launch follows, and the workspace
    // may still be read by it (programmatic dependent launch)
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t total = p.a_words + p.b_words;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    bool bad = false;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < total;
         w += stride) {
        if (w < p.a_words) {
            const int64_t tk = w >> 7;              // (tile, step)
            const int pos = static_cast<int>(w & 127);
            const int64_t t = tk / p.steps;
            const int ks = static_cast<int>(tk - t * p.steps);
            const int r = (pos & 3) * 32 + (pos >> 2);
            int64_t m, sa_goff = 0;
            int g = 0;
            if (p.masked) {
                g = static_cast<int>(t / p.tiles_per_group);
                m = (t - static_cast<int64_t>(g) * p.tiles_per_group) * kBM + r;
                sa_goff = static_cast<int64_t>(g) * p.sa_g_stride;
            } else {
                m = t * kBM + r;
            }
            // images of masked tiles that no unit reads (past masked_m[g]) are not
            // written
            bool used, stored = false;
            if (p.masked) {
                int mm = __ldg(p.row_info + g);
                mm = mm < 0 ? 0 : (mm > p.rows ? static_cast<int>(p.rows) : mm);
                const int64_t tile_m0 = (t - static_cast<int64_t>(g) * p.tiles_per_group) * kBM;
                used = tile_m0 < mm || (tile_m0 >= kBM && tile_m0 - kBM < mm);  // or a pair's idle half
                stored = m < mm;
            } else {
                const int tg = __ldg(p.row_info + t * kBM);
                used = true;  // the idle half of an odd pair reads the tile after it
                stored = m < p.rows && tg >= 0 && __ldg(p.row_info + m) == tg;
            }
            if (!used) continue;
            uint32_t code[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int kb = 2 * ks + j;
                uint32_t v = 0;
                if (m < p.rows && kb < p.kb_count) {
                    v = __float_as_uint(
                        __ldg(p.sa + sa_goff + kb * p.sa_kb_stride + m * p.sa_row_stride));
                    bad |= stored && !ue8m0_scale_ok(v);
                }
                code[j] = ue8m0_code(v);
            }
            p.packed_a[w] = code[0] | (code[1] << 8) | (code[0] << 16) | (code[1] << 24);
        } else {
            const int64_t wb = w - p.a_words;
            const int64_t ck = wb >> 7;             // (g * N/128 + nb, step)
            const int64_t c = ck / p.steps;
            const int ks = static_cast<int>(ck - c * p.steps);
            uint32_t code[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int kb = 2 * ks + j;
                code[j] = kb < p.kb_count ? ue8m0_code(__float_as_uint(__ldg(p.sb + c * p.kb_count + kb)))
                                          : 0u;
            }
            p.packed_b[wb] = code[0] | (code[1] << 8) | (code[0] << 16) | (code[1] << 24);
        }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) raise_error(p.err, kErrBadScale);
}

}  // namespace fp8bs
