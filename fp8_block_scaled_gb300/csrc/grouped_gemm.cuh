// Persistent grouped FP8 (E4M3) block-scaled GEMM for sm_103a.
//
// Operation (FlyDSL PR #433 "Adds Grouped and Batched GEMM kernels with
// blockscaling matching DeepGEMM API", section Summary):
//   D[r, n] = sum_kb sa[r, kb] * sb[g, n/128, kb] * (A[r, kb-block] . B[g, n, kb-block])
// with UE8M0 power-of-two scales that the matrix instruction applies
// (section "DeepGEMM conformance details": hardware E8M0 scaling path).
//
// One CTA per SM walks a static tile list (tile = 128 rows x BN columns).
// Warp roles inside a CTA of 256 threads:
//   warp 0      producer: per 128-K block, TMA loads of the A tile and the B
//               tile into a STAGES-deep shared-memory ring (complete on
//               full[stage]), plus 4-byte cp.async loads of the 128 activation
//               scales and BN/128 weight scales of that block (complete on
//               sf_raw[stage]).
//   warp 3      scale converter: turns the raw fp32 scales into UE8M0 bytes
//               laid out for tcgen05.cp and signals sf_ready[stage].
//   warp 1      MMA issuer: copies the stage's scales to TMEM, issues four
//               K=32 kind::mxf8f6f4 block-scaled MMAs into the fp32 TMEM
//               accumulator, and commits the stage back to the producer.
//   warp 2      allocates / frees the tensor memory.
//   warps 4-7   epilogue: TMEM -> registers (64 columns per load) ->
//               bf16/f16 (round to nearest even) -> 16-byte stores of the
//               valid rows; the accumulator is released to the MMA warp as
//               soon as its last columns are in registers.
// Every mbarrier wait is bounded in time; a wait that gives up records
// FP8BS_DEVERR_TIMEOUT, and the CTA drains its copies and MMAs, frees its
// tensor memory and exits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fp8bs {

constexpr int kBM = 128;            // rows per tile (MMA M)
constexpr int kBK = 128;            // K per stage = one scale block = 128 B of E4M3
constexpr int kUmmaK = 32;          // K per MMA instruction for 8-bit operands
constexpr int kThreads = 256;
constexpr int kMaxMaskedGroups = 1024;
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s per wait

constexpr uint32_t kErrTimeout = 0x1u;
constexpr uint32_t kErrMaskedM = 0x2u;
constexpr uint32_t kErrMixedTile = 0x4u;
constexpr uint32_t kErrBadGroup = 0x8u;
constexpr uint32_t kErrBadScale = 0x10u;
// GemmParams::debug_flags (test hook, 0 in normal use): the CTA-pair kernel's
// MMA thread first waits on a barrier nothing arrives on, so its bounded wait
// runs out and the launch takes the abort path.
constexpr uint32_t kDebugStallMma = 0x1u;

struct GemmParams {
    const float* sa;             // activation scales
    const float* sb;             // weight scales [G, N/128, K/128]
    const int32_t* row_info;     // contiguous: grouped_layout [m_sum]; masked: masked_m [G]
    void* d;                     // output
    uint32_t* err;               // device error word
    int64_t rows;                // contiguous: m_sum; masked: m_max
    int64_t sa_g_stride;         // elements between groups (masked KM / MK), 0 for contiguous
    int64_t sa_kb_stride;        // elements between K-blocks
    int64_t sa_row_stride;       // elements between rows
    int n, k, num_groups, kb_count, nb_count;
    int num_m_tiles;             // contiguous: ceil(m_sum/128); masked: ceil(m_max/128)
    int num_n_tiles;
    int raster_band;             // contiguous: m-tiles per rasterisation band
    // stream-K tail of the CTA-pair kernel (sk_slots == 0 disables it)
    float* sk_partial;           // sk_slots x [128 rows x 256 cols] fp32 partial accumulators
    uint32_t* sk_flags;          // 2 words per slot (ready tail warps; spare), 0 between launches
    int sk_slots;                // slots available (needs 2 per CTA pair of the grid)
    // fused gate/up epilogue of the CTA-pair kernel: d receives E4M3 codes [rows, n/2],
    // q_scale one fp32 UE8M0 scale per row and 128-column block
    float* q_scale;
    int64_t qs_g_stride;         // masked: elements between groups; contiguous: 0
    int64_t qs_row_stride;       // elements between rows
    int64_t qs_col_stride;       // elements between 128-column blocks
    uint32_t debug_flags;        // kDebug* test hooks, 0 in normal use
    int* list_ws;                // pair kernels: device pair list (list_ws_stride ints per
                                 // CTA) when it outgrows shared memory, else null
    int list_ws_stride;
    int d_align16;               // pair kernel: d is 16- but not 32-byte aligned (16-byte stores)
    int n_half;                  // pair kernel: n % 256 == 128, the last column tile is 128 wide
    // pair kernel, E4M3: the scale images of scale_pack_kernel (null: the kernel gathers
    // and converts the fp32 scales itself), with sf_steps pipeline steps per unit
    const uint32_t* sf_a_packed;
    const uint32_t* sf_b_packed;
    int sf_steps;
};

template <int BN>
struct SmemLayout {
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr int kABytes = kBM * kBK;           // 16 KB
    static constexpr int kBBytes = BN * kBK;
    static constexpr int kSfaBytes = 512;               // 128 words, tcgen05.cp order
    static constexpr int kSfbBytes = (BN / 128) * 512;
    static constexpr int kSaRawBytes = kBM * 4;
    static constexpr int kSbRawBytes = 16;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kABytes;
    static constexpr int kOffSfa = kOffB + kStages * kBBytes;
    static constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
    static constexpr int kOffSaRaw = kOffSfb + kStages * kSfbBytes;
    static constexpr int kOffSbRaw = kOffSaRaw + kStages * kSaRawBytes;
    static constexpr int kOffBar = (kOffSbRaw + kStages * kSbRawBytes + 7) / 8 * 8;
    // full[S], empty[S], sf_raw[S], sf_ready[S], tmem_full, tmem_empty, drain
    static constexpr int kNumBars = 4 * kStages + 3;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag
    static constexpr int kOffPrefix = kOffMisc + 16;
    static constexpr int kBytesContiguous = kOffPrefix;
    static constexpr int kBytesMasked = kOffPrefix + (kMaxMaskedGroups + 1) * 4;
    static constexpr int kAlignSlack = 1024;
    // TMEM: accumulator in columns [0, BN), then per stage 4 columns of
    // activation scales and BN/32 columns of weight scales.
    static constexpr int kSfCols = 4 + BN / 32;
    static constexpr int kTmemColsUsed = BN + kStages * kSfCols;
    static constexpr int kTmemCols = kTmemColsUsed <= 256 ? 256 : 512;
    static_assert(kTmemColsUsed <= 512, "TMEM budget");
    static_assert(kOffB % 1024 == 0, "B tiles must stay 1024-aligned");
    static_assert(kBytesMasked + kAlignSlack <= 232448, "shared memory budget");
};

struct Tile {
    int g;        // group; < 0 means skip
    int m_tile;   // 128-row tile index (global for contiguous, within group for masked)
    int n_tile;
};

__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t bits) {
    atomicOr(err, bits);
}

// Bounded wait on an mbarrier phase.  Returns false when the CTA is aborting
// (another role gave up) or when this wait exceeded the limit.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           uint32_t* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            raise_error(err, kErrTimeout);
            return false;
        }
    }
}

// Whole-warp wait: every lane waits, the result is the AND over lanes.
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity,
                                                volatile int* abort_flag, uint32_t* err) {
    bool ok = wait_phase(bar, parity, abort_flag, err);
    return __all_sync(0xffffffffu, ok);
}

// Contiguous variant: tile t -> (m_tile, n_tile) with grouped-M rasterisation
// (bands of `raster_band` m-tiles walked column-major so that concurrently
// running CTAs share B tiles in L2).  The first row of a 128-row tile names
// its group (the contiguous layout pads every expert to a multiple of 128
// rows); a tile whose first row is -1 is skipped.  Warp-uniform: every lane
// computes the same tile.
__device__ __forceinline__ Tile contiguous_tile(const GemmParams& p, int t, bool report) {
    const int band_tiles = p.raster_band * p.num_n_tiles;
    const int band = t / band_tiles;
    const int r = t - band * band_tiles;
    const int m_base = band * p.raster_band;
    const int gm = min(p.raster_band, p.num_m_tiles - m_base);
    Tile tile;
    tile.m_tile = m_base + r % gm;
    tile.n_tile = r / gm;
    int v = __ldg(p.row_info + static_cast<int64_t>(tile.m_tile) * kBM);
    if (v >= p.num_groups || v < -1) {
        if (report && (threadIdx.x & 31) == 0) raise_error(p.err, kErrBadGroup);
        v = -1;
    }
    tile.g = v;
    return tile;
}

// Masked variant: tiles are ordered (group, n_tile, m_tile) with m fastest, so
// the m-tiles that share one B tile run on neighbouring CTAs.  prefix[g] is the
// number of tiles before group g (shared memory).
__device__ __forceinline__ Tile masked_tile(const GemmParams& p, const int* prefix, int t) {
    int lo = 0, hi = p.num_groups;  // find g with prefix[g] <= t < prefix[g+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= t) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int local = t - prefix[g];
    const int mt = (prefix[g + 1] - prefix[g]) / p.num_n_tiles;
    Tile tile;
    tile.g = g;
    tile.n_tile = local / mt;
    tile.m_tile = local - tile.n_tile * mt;
    return tile;
}

template <typename OutT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);

template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Whether an fp32 scale is a UE8M0 value: a positive power of two whose
// exponent field the scale converters can take as the scale byte -- a normal
// power of two (mantissa zero, exponent field 1..254, i.e. 2^-126..2^127) or
// 2^-127, whose fp32 form is the subnormal 0x00400000 and whose exponent field
// is 0, the UE8M0 code of 2^-127.  Anything else (another value, zero, a
// negative or subnormal number, inf, NaN) would be truncated to a different
// scale, so a stored row that reads one raises kErrBadScale.
__device__ __forceinline__ bool ue8m0_scale_ok(uint32_t fbits) {
    return ((fbits & 0x807FFFFFu) == 0u && fbits - 0x00800000u < 0x7F000000u) ||
           fbits == 0x00400000u;
}

// fp32 power-of-two scale -> its exponent byte (the UE8M0 code), repeated in
// all four bytes so that any scale-factor byte selector reads it.
__device__ __forceinline__ uint32_t ue8m0_x4(uint32_t fbits) {
    return ((fbits >> 23) & 0xFFu) * 0x01010101u;
}

template <int BN, typename OutT, bool kMasked>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
    using L = SmemLayout<BN>;
    constexpr int S = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto bar_full = [&](int s) { return sbase + L::kOffBar + 8u * s; };
    auto bar_empty = [&](int s) { return sbase + L::kOffBar + 8u * (S + s); };
    auto bar_sf_raw = [&](int s) { return sbase + L::kOffBar + 8u * (2 * S + s); };
    auto bar_sf_ready = [&](int s) { return sbase + L::kOffBar + 8u * (3 * S + s); };
    const uint32_t bar_tmem_full = sbase + L::kOffBar + 8u * (4 * S);
    const uint32_t bar_tmem_empty = sbase + L::kOffBar + 8u * (4 * S + 1);
    const uint32_t bar_drain = sbase + L::kOffBar + 8u * (4 * S + 2);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
    int* prefix = reinterpret_cast<int*>(smem + L::kOffPrefix);

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full(s), 1);       // producer arrive.expect_tx (+ TMA bytes)
            mbar_init(bar_empty(s), 1);      // tcgen05.commit
            mbar_init(bar_sf_raw(s), 32);    // one cp.async arrival per producer lane
            mbar_init(bar_sf_ready(s), 1);   // scale converter
        }
        mbar_init(bar_tmem_full, 1);
        mbar_init(bar_tmem_empty, 4);        // one arrival per epilogue warp
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
    }
    // inputs, outputs and the error word may belong to the grid this launch
    // follows (programmatic dependent launch): wait for it before touching them
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp == 2) {
        tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
        tmem_relinquish();
    }
    int total_tiles;
    if constexpr (kMasked) {
        // per-group tile counts and their exclusive prefix (warp 3 scans)
        if (warp == 3) {
            const int G = p.num_groups;
            const int per = (G + 31) / 32;
            const int g0 = lane * per;
            int local = 0;
            for (int g = g0; g < min(G, g0 + per); ++g) {
                int mm = __ldg(p.row_info + g);
                if (mm < 0 || mm > p.rows) {
                    raise_error(p.err, kErrMaskedM);
                    mm = mm < 0 ? 0 : static_cast<int>(p.rows);
                }
                local += (mm + kBM - 1) / kBM * p.num_n_tiles;
            }
            int incl = local;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            int run = incl - local;
            for (int g = g0; g < min(G, g0 + per); ++g) {
                prefix[g] = run;
                int mm = __ldg(p.row_info + g);
                mm = mm < 0 ? 0 : (mm > p.rows ? static_cast<int>(p.rows) : mm);
                run += (mm + kBM - 1) / kBM * p.num_n_tiles;
            }
            if (lane == 31) prefix[G] = incl;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if constexpr (kMasked) {
        total_tiles = prefix[p.num_groups];
    } else {
        total_tiles = p.num_m_tiles * p.num_n_tiles;
    }

    auto get_tile = [&](int t, bool report) -> Tile {
        if constexpr (kMasked) {
            return masked_tile(p, prefix, t);
        } else {
            return contiguous_tile(p, t, report);
        }
    };

    constexpr uint32_t kTxBytes = (kBM + BN) * kBK;
    constexpr uint32_t kIdesc = make_idesc_mxf8(kBM, BN);
    constexpr uint32_t kAccCol = 0;
    const int KB = p.kb_count;

    if (warp == 0) {
        // ============================================================ producer
        int s = 0;
        uint32_t ph = 0;
        uint32_t issued_mask = 0;           // stages holding copies this warp issued
        uint32_t issued_parity = 0;         // parity of the last phase issued per stage
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            const Tile tile = get_tile(t, true);
            if (tile.g < 0) continue;
            int64_t a_row0, m_base;
            int64_t sa_goff = 0;
            if constexpr (kMasked) {
                m_base = static_cast<int64_t>(tile.m_tile) * kBM;
                a_row0 = static_cast<int64_t>(tile.g) * p.rows + m_base;
                sa_goff = static_cast<int64_t>(tile.g) * p.sa_g_stride;
            } else {
                m_base = static_cast<int64_t>(tile.m_tile) * kBM;
                a_row0 = m_base;
            }
            const int b_row0 = tile.g * p.n + tile.n_tile * BN;
            const int nb0 = tile.n_tile * (BN / 128);
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait_phase(bar_empty(s), ph ^ 1u, abort_flag, p.err)) { ok = false; break; }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar_full(s), kTxBytes);
                    tma_load_2d(sbase + L::kOffA + s * L::kABytes, &tmap_a, kb * kBK,
                                static_cast<int32_t>(a_row0), bar_full(s));
                    tma_load_2d(sbase + L::kOffB + s * L::kBBytes, &tmap_b, kb * kBK, b_row0,
                                bar_full(s));
                }
                const uint32_t sa_dst = sbase + L::kOffSaRaw + s * L::kSaRawBytes;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = j * 32 + lane;
                    const int64_t m = m_base + r;
                    const bool in = m < p.rows;
                    const float* src = p.sa + sa_goff + kb * p.sa_kb_stride + m * p.sa_row_stride;
                    cp_async_4(sa_dst + 4u * r, in ? src : p.sa, in ? 4u : 0u);
                }
                if (lane < BN / 128) {
                    const float* src =
                        p.sb + (static_cast<int64_t>(tile.g) * p.nb_count + nb0 + lane) * KB + kb;
                    cp_async_4(sbase + L::kOffSbRaw + s * L::kSbRawBytes + 4u * lane, src, 4u);
                }
                cp_async_mbar_arrive_noinc(bar_sf_raw(s));
                issued_mask |= 1u << s;
                issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                if (++s == S) { s = 0; ph ^= 1u; }
            }
        }
        if (!ok) {
            // let every copy already in flight land before the CTA goes away
            for (int i = 0; i < S; ++i) {
                if (issued_mask & (1u << i)) {
                    const uint32_t par = (issued_parity >> i) & 1u;
                    const uint64_t t0 = global_timer_ns();
                    while (!(mbar_try_wait(bar_full(i), par) && mbar_try_wait(bar_sf_raw(i), par)) &&
                           global_timer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        int s = 0;
        uint32_t ph = 0, acc_ph = 0;
        bool ok = true;
        bool issued_any = false;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            const Tile tile = get_tile(t, false);
            if (tile.g < 0) continue;
            if (!warp_wait_phase(bar_tmem_empty, acc_ph ^ 1u, abort_flag, p.err)) { ok = false; break; }
            tc_fence_after();
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait_phase(bar_full(s), ph, abort_flag, p.err) ||
                    !warp_wait_phase(bar_sf_ready(s), ph, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sf_col = BN + s * L::kSfCols;
                    tc_cp_32x128b_warpx4(tmem_base + sf_col,
                                         make_desc_sf(sbase + L::kOffSfa + s * L::kSfaBytes));
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j) {
                        tc_cp_32x128b_warpx4(
                            tmem_base + sf_col + 4 + 4 * j,
                            make_desc_sf(sbase + L::kOffSfb + s * L::kSfbBytes + 512 * j));
                    }
                    const uint64_t adesc = make_desc_sw128(sbase + L::kOffA + s * L::kABytes);
                    const uint64_t bdesc = make_desc_sw128(sbase + L::kOffB + s * L::kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        // advance the start address by k*32 bytes inside the swizzle atom
                        tc_mma_mxf8(tmem_base + kAccCol, adesc + 2u * k, bdesc + 2u * k, kIdesc,
                                    tmem_base + sf_col, tmem_base + sf_col + 4,
                                    (kb | k) != 0 ? 1u : 0u);
                    }
                    tc_commit(bar_empty(s));
                }
                issued_any = true;
                __syncwarp();
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(bar_tmem_full);
            acc_ph ^= 1u;
        }
        if (!ok && issued_any) {
            // wait until every MMA this thread issued has finished with TMEM
            if (lane == 0) {
                tc_commit(bar_drain);
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar_drain, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
            __syncwarp();
        }
    } else if (warp == 3) {
        // ============================================================ scale converter
        // raw fp32 scales (row order) -> UE8M0 words in tcgen05.cp order:
        // word (lane*4 + c) holds row 32*c + lane; weight scales replicated
        // over their 128 columns.
        // The scales of every row whose result is stored, and the tile's weight
        // scales, are checked to be UE8M0 values (ue8m0_scale_ok); rows that are
        // not computed may hold anything.
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        bool bad = false;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            const Tile tile = get_tile(t, false);
            if (tile.g < 0) continue;
            uint32_t live = 0;  // bit q: row 32 q + lane of the tile is stored
            int mm = 0;
            if constexpr (kMasked) {
                mm = __ldg(p.row_info + tile.g);
                mm = mm < 0 ? 0 : (mm > p.rows ? static_cast<int>(p.rows) : mm);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t m = static_cast<int64_t>(tile.m_tile) * kBM + q * 32 + lane;
                bool stored;
                if constexpr (kMasked) stored = m < mm;
                else stored = m < p.rows && __ldg(p.row_info + m) == tile.g;
                live |= stored ? 1u << q : 0u;
            }
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait_phase(bar_sf_raw(s), ph, abort_flag, p.err)) { ok = false; break; }
                const uint32_t* raw = reinterpret_cast<const uint32_t*>(
                    smem + L::kOffSaRaw + s * L::kSaRawBytes);
                uint4 w;
                w.x = ue8m0_x4(raw[lane]);
                w.y = ue8m0_x4(raw[32 + lane]);
                w.z = ue8m0_x4(raw[64 + lane]);
                w.w = ue8m0_x4(raw[96 + lane]);
                *reinterpret_cast<uint4*>(smem + L::kOffSfa + s * L::kSfaBytes + 16 * lane) = w;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    bad |= ((live >> q) & 1u) != 0u && !ue8m0_scale_ok(raw[32 * q + lane]);
                const uint32_t* sbraw = reinterpret_cast<const uint32_t*>(
                    smem + L::kOffSbRaw + s * L::kSbRawBytes);
#pragma unroll
                for (int j = 0; j < BN / 128; ++j) {
                    const uint32_t v = ue8m0_x4(sbraw[j]);
                    *reinterpret_cast<uint4*>(smem + L::kOffSfb + s * L::kSfbBytes + 512 * j +
                                              16 * lane) = make_uint4(v, v, v, v);
                }
                bad |= lane < BN / 128 && !ue8m0_scale_ok(sbraw[lane < BN / 128 ? lane : 0]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sf_ready(s));
                if (++s == S) { s = 0; ph ^= 1u; }
            }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(p.err, kErrBadScale);
    } else if (warp >= 4) {
        // ============================================================ epilogue
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int row_in_tile = q * 32 + lane;
        uint32_t acc_ph = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
            const Tile tile = get_tile(t, false);
            if (tile.g < 0) continue;
            // row validity and destination, resolved before the accumulator is ready
            bool valid;
            int64_t drow;
            if constexpr (kMasked) {
                const int64_t m = static_cast<int64_t>(tile.m_tile) * kBM + row_in_tile;
                int mm = __ldg(p.row_info + tile.g);
                mm = mm < 0 ? 0 : (mm > p.rows ? static_cast<int>(p.rows) : mm);
                valid = m < mm;
                drow = static_cast<int64_t>(tile.g) * p.rows + m;
            } else {
                drow = static_cast<int64_t>(tile.m_tile) * kBM + row_in_tile;
                const int lv = drow < p.rows ? __ldg(p.row_info + drow) : -1;
                valid = lv == tile.g;
                if (!valid) {
                    if (lv >= p.num_groups || lv < -1) raise_error(p.err, kErrBadGroup);
                    else if (lv >= 0) raise_error(p.err, kErrMixedTile);
                }
            }
            if (!warp_wait_phase(bar_tmem_full, acc_ph, abort_flag, p.err)) break;
            tc_fence_after();
            OutT* out = static_cast<OutT*>(p.d) + drow * p.n + tile.n_tile * BN;
            constexpr int kChunk = 64;
#pragma unroll 1
            for (int c = 0; c < BN / kChunk; ++c) {
                uint32_t v[kChunk];
                tc_ld_32x32b_x64_sync(
                    tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + c * kChunk, v);
                if (c == BN / kChunk - 1) {
                    // the whole accumulator is in registers: hand TMEM back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_tmem_empty);
                }
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(out + c * kChunk);
#pragma unroll
                    for (int i = 0; i < kChunk / 8; ++i) {
                        dst[i] = make_uint4(
                            pack2<OutT>(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1])),
                            pack2<OutT>(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                            pack2<OutT>(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                            pack2<OutT>(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
                    }
                }
            }
            acc_ph ^= 1u;
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem_base, L::kTmemCols);
}

}  // namespace fp8bs
