// CTA-pair (cluster of 2) variant of the grouped FP8 block-scaled GEMM.
//
// Same operation as grouped_gemm.cuh ("Adds Grouped and Batched GEMM kernels
// with blockscaling matching DeepGEMM API", FlyDSL PR #433, section Summary),
// computed in 256 x 256 output tiles by a pair of CTAs on two SMs: each CTA
// holds 128 rows of A and 128 of the tile's 256 rows of B in shared memory and
// owns a 128 x 256 fp32 accumulator in its tensor memory; the leader CTA
// (cluster rank 0) issues tcgen05.mma.cta_group::2 with M = 256, N = 256, so
// each SM streams 32 KB of operands per 128-K block instead of 48 KB.
//
// Contiguous variant: a pair of 128-row tiles must belong to one expert, so
// the kernel first scans grouped_layout (one row per 128-row tile, the rule
// of the contiguous layout: the first row of a tile names its expert, -1
// skips the tile) and pairs the tiles of every expert segment two by two; an
// odd last tile runs with the second CTA idle-storing.  Masked variant: each
// group's first masked_m[g] rows are covered by ceil(masked_m[g] / 256) pairs.
//
// Scheduling: units (one 256 x 256 tile each) go round-robin to the pairs of
// the persistent grid.  When the unit count is not a multiple of the pair
// count, the units of the last two rounds are instead cut into equal runs of
// K steps, one contiguous run per pair (stream-K): every unit is then split at
// most once, into a head [0, x) finished last by one pair and a tail [x, end)
// finished first by the next pair.  Each epilogue warp of the tail writes its
// rows of the fp32 partial accumulator to a scratch slot and counts itself in
// the slot's ready word.  The head is always its pair's last piece, so the two
// ring stages after its last step are never loaded again: the A producer waits
// for their MMAs to release them, waits (bounded) until all four tail warps
// have counted themselves, and copies the 128 KB slot into them with four
// bulk copies that overlap the head's last steps; every epilogue warp then
// adds the partial chunk by chunk from shared memory, and one resets the ready
// word for the next launch.  Reading the partial with plain loads instead left
// four dependent round trips to a remote L2 slice exposed at the very end of
// the kernel.
//
// Operand staging: each pipeline stage holds two 128-K blocks, fetched with
// one 3-D TMA box per operand (128 bytes x 128 rows x 2 blocks); the A and B
// boxes are issued by two different warps.  One thread issues at most a few
// million boxes a second whatever their size, so large boxes from two issuers
// keep the issue rate well below that while 64 KB per stage is in flight.  In
// a masked unit whose second 128 rows all lie past masked_m[g], the peer CTA
// fetches no A at all (those rows of the product are never stored).
//
// Warp roles per CTA (both CTAs run all roles except the MMA issue):
//   warp 0  A producer: TMA of its 128 rows of A (completion counted on the
//           leader's full barrier, which only the leader arms, for the bytes
//           of both CTAs), cp.async of the raw fp32 scales
//   warp 2  B producer (after allocating the pair's tensor memory)
//   warp 3  scale converter: UE8M0 scale words in tcgen05.cp order, one word
//           per row (SFA) or column chunk (SFB) and stage with byte j for the
//           stage's K block j, then an arrival on the leader's full barrier
//   warp 1  (leader only, one thread) tcgen05.cp / tcgen05.mma issue,
//           commits multicast to both CTAs.  Scale copies take tensor-pipe
//           time, so they are issued once per stage; the MMAs of K block j
//           select byte j of the words through their scale ids.
//   warps 4-7 epilogue of the CTA's own 128 rows
//
// Fused gate/up epilogue (kSwiglu): for the first MoE GEMM, whose B holds the
// gate rows [0, N/2) and the up rows [N/2, N) of each expert, a unit covers
// 128 output columns j0..j0+127: the leader CTA loads gate rows j0.., the peer
// up rows N/2+j0.., so each CTA's accumulator holds gate in columns 0-127 and
// up in 128-255 for its 128 rows.  Each epilogue thread owns one row: it forms
// h = SiLU(gate) * up for the 128 columns ("flydsl mxfp4 a4w4 MoE: bring
// gemm1/gemm2 to parity with the HIP backend", section gemm1, silu_mul with
// the hardware exponential), takes the block's amax, the UE8M0 ceil scale of
// amax / 448 and the round-to-nearest-even E4M3 codes of h / scale (the
// quantiser of "Adds Grouped and Batched GEMM kernels with blockscaling
// matching DeepGEMM API", DeepGEMM conformance details), and stores 128 code
// bytes and one fp32 scale: the input format of the down projection.
#pragma once

#include "grouped_gemm.cuh"

namespace fp8bs {

constexpr int kPairMaxTiles = 4096;  // contiguous: 128-row tiles the shared-memory list holds
// contiguous, with the pair list in a device workspace: the prologue's layout
// scan indexes the operand stages as 4-byte entries (192 KB), and an entry holds
// a 16-bit tile index
constexpr int kPairMaxTilesWs = 32768;    // m_sum <= 4194304
constexpr int kPairMaxGroups = 1 << 15;   // expert ids of a pair-list entry
constexpr int kMxMaxTiles = 3968;    // MXFP4 (larger scale staging): m_sum <= 507904

// Shared-memory plan of the CTA-pair kernel.  kMx selects the MXFP4 variant:
// a "K block" is then 128 bytes of packed E2M1 (256 elements) and its scales
// (one E8M0 byte per 32 elements) are staged by cp.async straight into the
// tcgen05.cp layout, without the fp32 -> UE8M0 conversion of the E4M3 path.
template <bool kMx>
struct PairLayoutT {
    static constexpr int kKbPerStage = 2;                // K blocks per pipeline stage
    static constexpr int kStages = 3;
    static constexpr int kTileBytes = 128 * kBK;         // 128 rows x one K block
    static constexpr int kAStageBytes = kKbPerStage * kTileBytes;
    static constexpr int kBStageBytes = kKbPerStage * kTileBytes;
    // per K block: SFA and SFB in tcgen05.cp order (32x128b matrices of 512 bytes)
    static constexpr int kSfaBytes = kMx ? 1024 : 512;   // MX: two scale words per row
    static constexpr int kSfbBytes = kMx ? 2048 : 1024;  // both 128-column chunks
    static constexpr int kSaRawBytes = kMx ? 0 : 512;    // E4M3 path: raw fp32 scales
    static constexpr int kSbRawBytes = kMx ? 0 : 16;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kAStageBytes;
    static constexpr int kOffSfa = kOffB + kStages * kBStageBytes;
    static constexpr int kOffSfb = kOffSfa + kStages * kKbPerStage * kSfaBytes;
    static constexpr int kOffSaRaw = kOffSfb + kStages * kKbPerStage * kSfbBytes;
    static constexpr int kOffSbRaw = kOffSaRaw + kStages * kKbPerStage * kSaRawBytes;
    static constexpr int kOffBar =
        (kOffSbRaw + kStages * kKbPerStage * kSbRawBytes + 7) / 8 * 8;
    // full[S], empty[S], sf_raw[S], tmem_full, tmem_empty, drain, partial[4]
    static constexpr int kPartChunks = 4;                   // stream-K partial, 64 columns each
    static constexpr int kPartChunkBytes = 128 * 64 * 4;
    static constexpr int kNumBars = 3 * kStages + 3 + kPartChunks;
    static constexpr int kPrefetchStages = 3;  // stages of A/B prefetched into L2 ahead of the ring
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // slot, abort, scan scratch
    static constexpr int kMiscBytes = 16 + 2 * 16 * 4;
    static constexpr int kOffList = (kOffMisc + kMiscBytes + 15) / 16 * 16;
    static constexpr int kMaxTiles = kMx ? kMxMaxTiles : kPairMaxTiles;
    static constexpr int kListEntries = kMaxTiles + 1;
    static constexpr int kBytes = kOffList + kListEntries * 4;
    static constexpr int kAlignSlack = 1024;
    static constexpr int kSfColsPerKb = kMx ? 8 + 16 : 4 + 8;
    static constexpr int kTmemCols = 512;
    static_assert(256 + kStages * kKbPerStage * kSfColsPerKb <= kTmemCols, "TMEM budget");
    static_assert(kKbPerStage <= 4, "E4M3 scale words hold one byte per K block of a stage");
    static_assert(kBytes + kAlignSlack <= 232448, "shared memory budget");
    static_assert(kPairMaxTiles * 4 <= kStages * kAStageBytes, "prologue scratch");
    static_assert(kPairMaxTilesWs * 4 <= kStages * (kAStageBytes + kBStageBytes) &&
                      kOffB == kOffA + kStages * kAStageBytes,
                  "prologue scratch of a workspace-sized list (A and B stages contiguous)");
    static_assert(kPartChunks == 4 && kAStageBytes == kPartChunkBytes &&
                      kBStageBytes == kPartChunkBytes && kStages >= 2,
                  "stream-K partial staging: chunks fill the A and B halves of two stages");
};
using PairLayout = PairLayoutT<false>;

// Contiguous pair-list entry: first 128-row tile (bits 0..15), "second tile not
// part of the pair" flag (bit 16), expert id (bits 17..31).
__device__ __forceinline__ uint32_t pack_pair(int t0, bool half, int g) {
    return static_cast<uint32_t>(t0) | (half ? 1u << 16 : 0u) | (static_cast<uint32_t>(g) << 17);
}

// SiLU with the hardware exponential and the approximate (reciprocal-based)
// division: a relative error of a few fp32 ulps, far below one E4M3 step.  The
// IEEE-rounded division doubled the fused kernel's time.  Below x = -87 the
// denominator exceeds 2^126 and the quotient is a signed zero (the exact value
// is below 1e-35 in magnitude).
__device__ __forceinline__ float silu_f32(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// Four fp32 values -> four E4M3 codes (round to nearest even, finite values
// saturated), x0 in the lowest byte.  cvt ...e4m3x2 puts its first source in
// the upper byte of the 16-bit result.
__device__ __forceinline__ uint32_t pack4_e4m3(float x0, float x1, float x2, float x3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// One row's 128 activations -> UE8M0 ceil scale of amax / 448 (amax at least
// 1e-4, so an all-zero block gets a finite scale) and E4M3 codes of h / scale.
// The scale is a power of two, so h * (1 / scale) is exact.
__device__ __forceinline__ void quantize_store_row(const float (&h)[128], uint8_t* qdst,
                                                   float* sdst, bool valid) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 128; ++i) amax = fmaxf(amax, fabsf(h[i]));
    amax = fmaxf(amax, 1e-4f);
    const uint32_t tb = __float_as_uint(__fdiv_rn(amax, 448.0f));
    const uint32_t e = ((tb >> 23) & 0xFFu) + ((tb & 0x7FFFFFu) != 0u ? 1u : 0u);
    const float inv = __uint_as_float((254u - e) << 23);
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
        w[i] = pack4_e4m3(h[4 * i] * inv, h[4 * i + 1] * inv, h[4 * i + 2] * inv,
                          h[4 * i + 3] * inv);
    if (valid) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            st_global_v8(qdst + 32 * i, w[8 * i], w[8 * i + 1], w[8 * i + 2], w[8 * i + 3],
                         w[8 * i + 4], w[8 * i + 5], w[8 * i + 6], w[8 * i + 7]);
        *sdst = __uint_as_float(e << 23);
    }
}

// Block-wide scans over one int per thread of an NW-warp block; scratch holds
// 2 * kMaxScanWarps ints (the max scan uses the first half, the sum the second).
constexpr int kMaxScanWarps = 16;

template <int NW>
__device__ __forceinline__ int block_exclusive_max(int v, int* scratch) {
    static_assert(NW <= kMaxScanWarps, "scan scratch");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl = max(incl, o);
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int prev = -1;
    for (int w = 0; w < warp; ++w) prev = max(prev, scratch[w]);
    const int up = __shfl_up_sync(0xffffffffu, incl, 1);
    const int excl = lane == 0 ? prev : max(prev, up);
    __syncthreads();
    return excl;
}

template <int NW>
__device__ __forceinline__ int block_exclusive_sum(int v, int* scratch, int* total) {
    static_assert(NW <= kMaxScanWarps, "scan scratch");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) scratch[kMaxScanWarps + warp] = incl;
    __syncthreads();
    int prev = 0, all = 0;
    for (int w = 0; w < NW; ++w) {
        if (w < warp) prev += scratch[kMaxScanWarps + w];
        all += scratch[kMaxScanWarps + w];
    }
    *total = all;
    const int excl = prev + incl - v;
    __syncthreads();
    return excl;
}

// Bounded wait on a local mbarrier (arrivals may come from the peer CTA, from
// TMA completion or from tcgen05.commit).  On time-out the CTA and its peer
// are told to abort.
__device__ __forceinline__ bool pair_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t peer_abort, uint32_t* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            st_shared_cluster_u32(peer_abort, 1u);
            raise_error(err, kErrTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ bool pair_warp_wait(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, uint32_t peer_abort,
                                               uint32_t* err) {
    bool ok = pair_wait(bar, parity, abort_flag, peer_abort, err);
    return __all_sync(0xffffffffu, ok);
}

// One run of K steps [ks0, ks1) of unit u executed by a pair.
struct PairPiece {
    int u;      // < 0: no more pieces
    int ks0, ks1;
    int kind;   // 0 whole unit, 1 head (adds the partial of the unit's tail), 2 tail
};

struct PairUnit {
    int g;        // group / expert
    int n_tile;   // 256-column tile
    int m_base;   // first row of this CTA's half (contiguous: global row; masked: row in group)
    bool store;   // this CTA's half belongs to the unit
    bool half_n;  // the last column tile of an n % 256 == 128 problem: 128 columns wide
};

// Work units of one launch, the same on every CTA: contiguous -- the pair list
// (two 128-row tiles of one expert segment per entry, pack_pair format) built
// from grouped_layout, times the column tiles; masked -- per group
// ceil(masked_m[g] / 256) row pairs times the column tiles, as an exclusive
// prefix in list[0..G].  `scratch` is shared memory that is idle during the
// prologue (kPairMaxTiles ints).  All NT threads of the block call this.
template <bool kMasked, int NT>
__device__ __forceinline__ int build_units(const GemmParams& p, uint8_t* scratch_smem, int* list,
                                           int* scan_scratch) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int total_units;
    if constexpr (!kMasked) {
        // ---- pair list: tiles of each expert segment, two by two
        const int T = p.num_m_tiles;
        int* E = reinterpret_cast<int*>(scratch_smem);
        // all of a round's grouped_layout reads are issued before the first is used
        // (one round covers a list that fits shared memory)
        constexpr int kLoads = (kPairMaxTiles + NT - 1) / NT;
        for (int base = 0; base < T; base += kLoads * NT) {
            int ev[kLoads];
#pragma unroll
            for (int j = 0; j < kLoads; ++j) {
                const int t = base + static_cast<int>(threadIdx.x) + j * NT;
                ev[j] = t < T ? __ldg(p.row_info + static_cast<int64_t>(t) * kBM) : -1;
            }
#pragma unroll
            for (int j = 0; j < kLoads; ++j) {
                const int t = base + static_cast<int>(threadIdx.x) + j * NT;
                if (t < T) {
                    int v = ev[j];
                    if (v >= p.num_groups || v < -1) {
                        raise_error(p.err, kErrBadGroup);
                        v = -1;
                    }
                    E[t] = v;
                }
            }
        }
        __syncthreads();
        const int chunk = (T + NT - 1) / NT;
        const int lo = min(T, static_cast<int>(threadIdx.x) * chunk);
        const int hi = min(T, lo + chunk);
        int last_start = -1;
        for (int t = lo; t < hi; ++t)
            if (t == 0 || E[t] != E[t - 1]) last_start = t;
        const int carry = block_exclusive_max<NT / 32>(last_start, scan_scratch);
        int start = carry, count = 0;
        for (int t = lo; t < hi; ++t) {
            if (t == 0 || E[t] != E[t - 1]) start = t;
            if (E[t] >= 0 && ((t - start) & 1) == 0) ++count;
        }
        int total = 0;
        int idx = block_exclusive_sum<NT / 32>(count, scan_scratch, &total);
        start = carry;
        for (int t = lo; t < hi; ++t) {
            if (t == 0 || E[t] != E[t - 1]) start = t;
            if (E[t] >= 0 && ((t - start) & 1) == 0) {
                const bool half = (t + 1 >= T) || (E[t + 1] != E[t]);
                list[idx++] = static_cast<int>(pack_pair(t, half, E[t]));
            }
        }
        total_units = total * p.num_n_tiles;
    } else {
        // ---- masked: pairs per group and their prefix (warp 3)
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
                local += (mm + 2 * kBM - 1) / (2 * kBM) * p.num_n_tiles;
            }
            int incl = local;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            int run = incl - local;
            for (int g = g0; g < min(G, g0 + per); ++g) {
                list[g] = run;
                int mm = __ldg(p.row_info + g);
                mm = mm < 0 ? 0 : (mm > p.rows ? static_cast<int>(p.rows) : mm);
                run += (mm + 2 * kBM - 1) / (2 * kBM) * p.num_n_tiles;
            }
            if (lane == 31) list[G] = incl;
        }
        __syncthreads();
        total_units = list[p.num_groups];
    }
    return total_units;
}

// Unit u -> (group, column tile, this CTA's 128-row half).  Contiguous units are
// rasterised in bands of 4 pair-list entries times all column tiles, column
// tile slowest within a band, so the B tiles of a band are reused from L2.
template <bool kMasked>
__device__ __forceinline__ PairUnit unit_of(const GemmParams& p, const int* list, int total_units,
                                            int u, uint32_t rank) {
    PairUnit w;
    if constexpr (!kMasked) {
        const int P = total_units / p.num_n_tiles;
        const int band_units = 4 * p.num_n_tiles;
        const int band = u / band_units;
        const int r = u - band * band_units;
        const int gp = min(4, P - band * 4);
        const int pi = band * 4 + r % gp;
        w.n_tile = r / gp;
        const uint32_t e = static_cast<uint32_t>(list[pi]);
        const int t0 = static_cast<int>(e & 0xFFFFu);
        const bool half = (e >> 16) & 1u;
        w.g = static_cast<int>(e >> 17);
        w.m_base = (t0 + static_cast<int>(rank)) * kBM;
        w.store = !(half && rank == 1);
    } else {
        int lo = 0, hi = p.num_groups;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (list[mid] <= u) lo = mid; else hi = mid;
        }
        const int local = u - list[lo];
        const int mp = (list[lo + 1] - list[lo]) / p.num_n_tiles;
        w.g = lo;
        w.n_tile = local / mp;
        w.m_base = (local - w.n_tile * mp) * 2 * kBM + static_cast<int>(rank) * kBM;
        w.store = true;
    }
    w.half_n = p.n_half != 0 && w.n_tile == p.num_n_tiles - 1;
    return w;
}

// L2 prefetch of a contiguous problem: the pairs working on one band share its A
// tiles (one per column tile) and its B tiles (one per row tile).  The same boxes
// prefetched by all of them flooded the L2 with duplicate misses, so only one
// unit prefetches each: for A the unit with column tile 0, for B the unit with
// the first row tile of its band -- in both cases the earliest of the sharers.
// Masked problems keep every unit prefetching: restricting them the same way
// (column tile 0 / a group's first row pair) made the masked workload 12% slower.
template <bool kMasked>
__device__ __forceinline__ bool prefetch_owner_of(const GemmParams& p, int total_units, int u,
                                                  bool is_a) {
    if constexpr (kMasked) {
        return true;
    } else {
        const int band_units = 4 * p.num_n_tiles;
        const int band = u / band_units;
        const int r = u - band * band_units;
        const int gp = min(4, total_units / p.num_n_tiles - band * 4);
        return is_a ? r < gp : r % gp == 0;
    }
}

template <typename OutT, bool kMasked, bool kSwiglu, bool kMx = false>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
    using L = PairLayoutT<kMx>;
    constexpr int S = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair_id = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    auto bar_full = [&](int s) { return sbase + L::kOffBar + 8u * s; };
    auto bar_empty = [&](int s) { return sbase + L::kOffBar + 8u * (S + s); };
    auto bar_sf_raw = [&](int s) { return sbase + L::kOffBar + 8u * (2 * S + s); };
    const uint32_t bar_tmem_full = sbase + L::kOffBar + 8u * (3 * S);
    const uint32_t bar_tmem_empty = sbase + L::kOffBar + 8u * (3 * S + 1);
    const uint32_t bar_drain = sbase + L::kOffBar + 8u * (3 * S + 2);
    auto bar_part = [&](int c) { return sbase + L::kOffBar + 8u * (3 * S + 3 + c); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
    int* scan_scratch = reinterpret_cast<int*>(smem + L::kOffMisc + 16);
    // the pair list: in shared memory, or this CTA's region of the device workspace
    int* list = p.list_ws != nullptr
                    ? p.list_ws + static_cast<int64_t>(blockIdx.x) * p.list_ws_stride
                    : reinterpret_cast<int*>(smem + L::kOffList);
    const uint32_t peer_abort = mapa_shared(smem_addr(smem + L::kOffMisc + 4), rank ^ 1u);

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // leader's A and B producers (arrive.expect_tx for both CTAs' bytes) + both
            // scale converters
            mbar_init(bar_full(s), 4);
            mbar_init(bar_empty(s), 1);      // leader's multicast commit
            // own A producer: 32 lanes' cp.async arrivals, or lane 1's arrival and the
            // bytes of its bulk copies of packed scale images
            mbar_init(bar_sf_raw(s), (!kMx && p.sf_a_packed != nullptr) ? 1 : 32);
        }
        mbar_init(bar_tmem_full, 1);
        mbar_init(bar_tmem_empty, 8);        // 4 epilogue warps x 2 CTAs
        mbar_init(bar_drain, 1);
        for (int c = 0; c < L::kPartChunks; ++c) mbar_init(bar_part(c), 1);  // one use per launch
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
    }
    // Everything above touches only this CTA and the kernel parameters; from
    // here on the inputs (and the outputs and scratch) may belong to the grid
    // this launch follows, so wait for it, then let a grid launched after this
    // one with programmatic serialization be scheduled onto the SMs this grid
    // frees (it waits for this grid's completion in its own wait).
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp == 2) {
        tmem_alloc_pair(smem_addr(tmem_slot), L::kTmemCols);
        tmem_relinquish_pair();
    }

    const int total_units = build_units<kMasked, kThreads>(p, smem + L::kOffA, list, scan_scratch);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // peer barriers initialised, tensor memory allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    auto get_unit = [&](int u) { return unit_of<kMasked>(p, list, total_units, u, rank); };

    constexpr uint32_t kIdesc = make_idesc_mxf8(2 * kBM, 256);
    constexpr uint32_t kIdescN128 = make_idesc_mxf8(2 * kBM, 128);  // 128-column tiles
    constexpr uint32_t kIdescMx0 = make_idesc_mxf4(2 * kBM, 256, 0);
    constexpr uint32_t kIdescMx2 = make_idesc_mxf4(2 * kBM, 256, 2);
    const int KB = p.kb_count;
    const int NKS = (KB + L::kKbPerStage - 1) / L::kKbPerStage;  // pipeline steps per unit
    bool aborted = false;

    // ---- schedule: round-robin units, then a stream-K tail (same on every thread)
    // Worth it when the idle share of the last round, spread over all rounds, is
    // above 10% (the partial tiles cost a few microseconds); the masked variant
    // (launched with sk_slots = 0) keeps the m-tiles of one B tile together.
    const int last_round = total_units % num_pairs;
    const int rounds = (total_units + num_pairs - 1) / num_pairs;
    const bool use_sk = p.sk_slots >= 2 * num_pairs && total_units > num_pairs && last_round != 0 &&
                        (num_pairs - last_round) * 10 > num_pairs * rounds;
    int dp_count, dp_units = 0, sk_begin = 0, sk_end = 0;
    if (use_sk) {
        dp_count = total_units / num_pairs - 1;
        dp_units = dp_count * num_pairs;
        const int64_t work = static_cast<int64_t>(total_units - dp_units) * NKS;
        sk_begin = static_cast<int>(work * pair_id / num_pairs);
        sk_end = static_cast<int>(work * (pair_id + 1) / num_pairs);
    } else {
        dp_count = pair_id < total_units ? (total_units - pair_id + num_pairs - 1) / num_pairs : 0;
    }
    auto get_piece = [&](int i) -> PairPiece {
        PairPiece pc;
        pc.u = -1;
        pc.ks0 = 0;
        pc.ks1 = NKS;
        pc.kind = 0;
        if (i < dp_count) {
            pc.u = pair_id + i * num_pairs;
            return pc;
        }
        if (!use_sk) return pc;
        int j = i - dp_count;
        int pos = sk_begin;
        while (pos < sk_end) {
            const int uu = pos / NKS;
            const int k0 = pos - uu * NKS;
            const int k1 = min(NKS, k0 + (sk_end - pos));
            if (j == 0) {
                pc.u = dp_units + uu;
                pc.ks0 = k0;
                pc.ks1 = k1;
                pc.kind = k0 > 0 ? 2 : (k1 < NKS ? 1 : 0);
                return pc;
            }
            --j;
            pos += k1 - k0;
        }
        return pc;
    };

    auto prefetch_owner = [&](int uu) {
        return prefetch_owner_of<kMasked>(p, total_units, uu, warp == 0);
    };

    // Masked: whether the 128 rows of group g starting at m0 hold a computed row.
    auto half_has_rows = [&](int g, int m0) {
        int mm = __ldg(p.row_info + g);
        mm = mm < 0 ? 0 : (mm > p.rows ? static_cast<int>(p.rows) : mm);
        return m0 < mm;
    };

    // First A / B row of this CTA for unit u.
    auto unit_rows = [&](const PairUnit& w, int64_t* a_row0, int* b_row0) {
        *a_row0 = kMasked ? static_cast<int64_t>(w.g) * p.rows + w.m_base
                          : static_cast<int64_t>(w.m_base);
        // fused gate/up: the leader holds gate rows, the peer the matching up rows; a
        // 128-column tile (half_n) gives each CTA 64 rows of B (its box loads 128, of
        // which the MMA reads the first 64)
        *b_row0 = kSwiglu ? w.g * p.n + static_cast<int>(rank) * (p.n >> 1) + w.n_tile * 128
                          : w.g * p.n + w.n_tile * 256 + static_cast<int>(rank) * (w.half_n ? 64 : 128);
    };

    if (warp == 0 || warp == 2) {
        // ============================================================ producers
        // warp 0: A boxes and the raw scales; warp 2: B boxes
        const bool is_a = warp == 0;
        const CUtensorMap* map = is_a ? &tmap_a : &tmap_b;
        const uint32_t op_off = is_a ? L::kOffA : L::kOffB;
        int s = 0;
        uint32_t ph = 0;
        int last_kind = 0;
        for (int pi = 0; !aborted; ++pi) {
            const PairPiece pc = get_piece(pi);
            if (pc.u < 0) break;
            const PairUnit w = get_unit(pc.u);
            int64_t a_row0;
            int b_row0;
            unit_rows(w, &a_row0, &b_row0);
            const int32_t row0 = is_a ? static_cast<int32_t>(a_row0) : b_row0;
            const int64_t sa_goff = kMasked ? static_cast<int64_t>(w.g) * p.sa_g_stride : 0;
            const int nb0 = w.n_tile * 2;
            // Masked: when the peer's 128 rows all lie at or past masked_m[g] (the last
            // pair of a group with masked_m % 256 in [1, 128]), the peer loads no A and the
            // leader arms for one CTA's A bytes.  The peer's stale A rows then enter the
            // MMA, but row r of the product depends only on row r of A, and those rows are
            // never stored.  Fewer L2 requests: about 2% on the masked decode workload.
            const bool peer_a_skip =
                kMasked && !kMx && !half_has_rows(w.g, w.m_base + (leader ? kBM : 0));
            const bool own_a_skip = is_a && !leader && peer_a_skip;
            for (int ks = pc.ks0; ks < pc.ks1; ++ks) {
                if (!pair_warp_wait(bar_empty(s), ph ^ 1u, abort_flag, peer_abort, p.err)) {
                    aborted = true;
                    break;
                }
                const int kb0 = ks * L::kKbPerStage;
                if (lane == 0) {
                    const uint32_t full_leader = mapa_shared(bar_full(s), 0);
                    // the leader arms its barrier for this operand's bytes of both CTAs; the
                    // peer's copies only complete into it
                    if (leader)
                        mbar_arrive_expect_tx(bar_full(s),
                                              (is_a && peer_a_skip ? 1u : 2u) * L::kAStageBytes);
                    if (!own_a_skip)
                        tma_load_3d_pair(sbase + op_off + s * L::kAStageBytes, map, 0, row0, kb0,
                                         full_leader);
                    // warm L2 with the box this warp loads kPrefetchStages steps later
                    // (the next piece's first steps near the end of this one)
                    int kp = ks + L::kPrefetchStages;
                    int32_t prow = row0;
                    bool pf = !own_a_skip && prefetch_owner(pc.u);
                    if (kp >= pc.ks1) {
                        const PairPiece np = get_piece(pi + 1);
                        pf = np.u >= 0 && prefetch_owner(np.u);
                        if (pf) {
                            int64_t na;
                            int nbr;
                            const PairUnit wn = get_unit(np.u);
                            unit_rows(wn, &na, &nbr);
                            prow = is_a ? static_cast<int32_t>(na) : nbr;
                            kp = np.ks0 + (kp - pc.ks1);
                            pf = kp < np.ks1 &&
                                 !(is_a && kMasked && !kMx && !half_has_rows(wn.g, wn.m_base));
                        }
                    }
                    if (pf) tma_prefetch_3d(map, 0, prow, kp * L::kKbPerStage);
                }
                if (is_a && !kMx && p.sf_a_packed != nullptr) {
                    // the stage's scale images, made by the scale pre-pass: 512 bytes of
                    // SFA for the CTA's 128 rows and 512 bytes for each of the unit's two
                    // weight-scale chunks, copied as they are (lane 1; lane 0 issues the
                    // operand box)
                    if (lane == 1) {
                        // a CTA half past the last tile (the idle half of an odd pair, or of a
                        // masked pair past m_max) copies the last tile's image: its rows are
                        // never stored
                        const int tl = min(w.m_base / kBM, p.num_m_tiles - 1);
                        const int64_t t = kMasked ? static_cast<int64_t>(w.g) * p.num_m_tiles + tl : tl;
                        const int gnb = w.g * p.nb_count;
                        const int c0 = kSwiglu ? w.n_tile : w.n_tile * 2;
                        // a 128-column tile has no second chunk: its image stands in (unused)
                        const int c1 = kSwiglu ? (p.n >> 8) + w.n_tile : min(w.n_tile * 2 + 1, p.nb_count - 1);
                        const uint32_t rb = bar_sf_raw(s);
                        mbar_arrive_expect_tx(rb, 3u * 512u);
                        bulk_load(sbase + L::kOffSfa + s * L::kKbPerStage * L::kSfaBytes,
                                  p.sf_a_packed + (t * p.sf_steps + ks) * 128, 512u, rb);
                        bulk_load(sbase + L::kOffSfb + s * L::kKbPerStage * L::kSfbBytes,
                                  p.sf_b_packed + (static_cast<int64_t>(gnb + c0) * p.sf_steps + ks) * 128,
                                  512u, rb);
                        bulk_load(sbase + L::kOffSfb + s * L::kKbPerStage * L::kSfbBytes + 512,
                                  p.sf_b_packed + (static_cast<int64_t>(gnb + c1) * p.sf_steps + ks) * 128,
                                  512u, rb);
                    }
                } else if (is_a && !kMx) {
                    // raw scales of the stage's K blocks (zero beyond K and past the rows)
#pragma unroll
                    for (int j = 0; j < L::kKbPerStage; ++j) {
                        const int kb = kb0 + j;
                        const uint32_t sa_dst =
                            sbase + L::kOffSaRaw + (s * L::kKbPerStage + j) * L::kSaRawBytes;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int r = q * 32 + lane;
                            const int64_t m = static_cast<int64_t>(w.m_base) + r;
                            const bool in = m < p.rows && kb < KB;
                            const float* src =
                                p.sa + sa_goff + kb * p.sa_kb_stride + m * p.sa_row_stride;
                            cp_async_4(sa_dst + 4u * r, in ? src : p.sa, in ? 4u : 0u);
                        }
                        if (lane < 2) {
                            // the two 128-column chunks of the unit's B tile (a 128-column
                            // tile has only the first; the second is zero)
                            const int nb = kSwiglu ? lane * (p.n >> 8) + w.n_tile : nb0 + lane;
                            const bool in = kb < KB && nb < p.nb_count;
                            const float* src =
                                p.sb + (static_cast<int64_t>(w.g) * p.nb_count + nb) * KB + kb;
                            cp_async_4(sbase + L::kOffSbRaw + (s * L::kKbPerStage + j) * L::kSbRawBytes +
                                           4u * lane,
                                       in ? src : p.sb, in ? 4u : 0u);
                        }
                    }
                    cp_async_mbar_arrive_noinc(bar_sf_raw(s));
                }
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            last_kind = pc.kind;
        }
        // The pair's last piece is the head of a split unit: copy the partial its tail
        // published into the two stages after the last step as soon as their MMAs
        // have completed (chunks 2j and 2j + 1 into the A and B halves of stage j),
        // so that the copies overlap the last steps instead of following them.
        if (is_a && last_kind == 1) {
            const int slot = (pair_id + 1) * 2 + static_cast<int>(rank);
            const float* src = p.sk_partial + static_cast<int64_t>(slot) * (128 * 256);
            for (int j = 0; j < 2 && !aborted; ++j) {
                if (!pair_warp_wait(bar_empty(s), ph ^ 1u, abort_flag, peer_abort, p.err)) {
                    aborted = true;
                    break;
                }
                if (lane == 0) {
                    if (j == 0) {
                        const uint64_t t0 = global_timer_ns();
                        while (ld_acquire_gpu_u32(p.sk_flags + 2 * slot) < 4u) {
                            if (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs) {
                                raise_error(p.err, kErrTimeout);
                                break;
                            }
                        }
                        // the copies are issued even after a time-out, so that no warp
                        // waits for them in vain (the error is already recorded)
                        fence_proxy_async_global();
                    }
                    for (int h = 0; h < 2; ++h) {
                        const int c = 2 * j + h;
                        mbar_arrive_expect_tx(bar_part(c), L::kPartChunkBytes);
                        bulk_load(sbase + (h ? L::kOffB + s * L::kBStageBytes
                                             : L::kOffA + s * L::kAStageBytes),
                                  src + c * (L::kPartChunkBytes / 4), L::kPartChunkBytes,
                                  bar_part(c));
                    }
                }
                __syncwarp();
                if (++s == S) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer (leader)
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0, acc_ph = 0;
            bool issued_any = false;
            // test hook: phase 0 of the drain barrier completes only after a drain commit,
            // which nothing has issued yet, so this wait runs out and the launch aborts
            if ((p.debug_flags & kDebugStallMma) &&
                !pair_wait(bar_drain, 0, abort_flag, peer_abort, p.err))
                aborted = true;
            for (int pi = 0; !aborted; ++pi) {
                const PairPiece pc = get_piece(pi);
                if (pc.u < 0) break;
                if (!pair_wait(bar_tmem_empty, acc_ph ^ 1u, abort_flag, peer_abort, p.err)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t idesc_unit =
                    (!kMx && p.n_half && get_unit(pc.u).half_n) ? kIdescN128 : kIdesc;
                for (int ks = pc.ks0; ks < pc.ks1; ++ks) {
                    if (!pair_wait(bar_full(s), ph, abort_flag, peer_abort, p.err)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < L::kKbPerStage; ++j) {
                        const int kb = ks * L::kKbPerStage + j;
                        if (kb >= KB) break;
                        if constexpr (kMx) {
                            const int slot = s * L::kKbPerStage + j;
                            const uint32_t sf_col = 256 + slot * L::kSfColsPerKb;
                            // SFA words 0, 1 -> columns +0, +4; SFB (word, N half) -> +8 + 4 * (2w + h)
#pragma unroll
                            for (int m = 0; m < 2; ++m)
                                tc_cp_pair_32x128b_warpx4(
                                    tmem_base + sf_col + 4 * m,
                                    make_desc_sf(sbase + L::kOffSfa + slot * L::kSfaBytes + 512 * m));
#pragma unroll
                            for (int m = 0; m < 4; ++m)
                                tc_cp_pair_32x128b_warpx4(
                                    tmem_base + sf_col + 8 + 4 * m,
                                    make_desc_sf(sbase + L::kOffSfb + slot * L::kSfbBytes + 512 * m));
                            const uint64_t adesc = make_desc_sw128(sbase + L::kOffA + s * L::kAStageBytes +
                                                                   j * L::kTileBytes);
                            const uint64_t bdesc = make_desc_sw128(sbase + L::kOffB + s * L::kBStageBytes +
                                                                   j * L::kTileBytes);
                            // MMA k covers elements 64k..64k+63 of the block: scale word k / 2,
                            // bytes 2 (k % 2) and 2 (k % 2) + 1 (the instruction's scale id)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc_mma_pair_mxf4(tmem_base, adesc + 2u * k, bdesc + 2u * k,
                                                 (k & 1) ? kIdescMx2 : kIdescMx0,
                                                 tmem_base + sf_col + 4 * (k >> 1),
                                                 tmem_base + sf_col + 8 + 8 * (k >> 1),
                                                 (ks > pc.ks0 || j > 0 || k > 0) ? 1u : 0u);
                            continue;
                        }
                        // the stage's scale words (byte j for K block j) are copied once, with
                        // its first K block, into the columns of the stage's first slot
                        const int slot0 = s * L::kKbPerStage;
                        const uint32_t sf0 = 256 + slot0 * L::kSfColsPerKb;
                        if (j == 0) {
                            tc_cp_pair_32x128b_warpx4(
                                tmem_base + sf0, make_desc_sf(sbase + L::kOffSfa + slot0 * L::kSfaBytes));
                            tc_cp_pair_32x128b_warpx4(
                                tmem_base + sf0 + 4,
                                make_desc_sf(sbase + L::kOffSfb + slot0 * L::kSfbBytes));
                            tc_cp_pair_32x128b_warpx4(
                                tmem_base + sf0 + 8,
                                make_desc_sf(sbase + L::kOffSfb + slot0 * L::kSfbBytes + 512));
                        }
                        const uint32_t idesc_j = idesc_scale_ids(idesc_unit, static_cast<uint32_t>(j));
                        const uint64_t adesc = make_desc_sw128(sbase + L::kOffA + s * L::kAStageBytes +
                                                               j * L::kTileBytes);
                        const uint64_t bdesc = make_desc_sw128(sbase + L::kOffB + s * L::kBStageBytes +
                                                               j * L::kTileBytes);
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k) {
                            // the first MMA of a piece overwrites the accumulator
                            tc_mma_pair_mxf8(tmem_base, adesc + 2u * k, bdesc + 2u * k, idesc_j,
                                             tmem_base + sf0, tmem_base + sf0 + 4,
                                             (ks > pc.ks0 || j > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    tc_commit_pair_mc(bar_empty(s), 0x3);
                    issued_any = true;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                if (aborted) break;
                tc_commit_pair_mc(bar_tmem_full, 0x3);
                acc_ph ^= 1u;
            }
            if (aborted && issued_any) {
                tc_commit_pair_mc(bar_drain, 0x1);
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar_drain, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 3 && kMx) {
        // ============================================================ MXFP4 scale staging
        // E8M0 bytes, [rows, K/32] for A (masked: per group, sa_g_stride bytes apart)
        // and [G*N, K/32] for B.  A K block has 8 per row = two 4-byte words; word w of
        // row r goes to lane r % 32, column r / 32 of 32x128b matrix w (SFB: matrix
        // 2w + n / 128), the layout tcgen05.cp moves into tensor memory unchanged.  This
        // warp issues a stage's copies as soon as the stage is free and signals the
        // stage one step later, so two stages of scales are in flight while the
        // producers issue only the operand boxes.
        //
        // When a scale row's stage slice (2 K blocks = 16 bytes) is 16-byte aligned
        // (K % 512 == 0), each row is fetched with one 16-byte copy into row-major
        // staging at the slot's own address, then rearranged in place: lane l fetches
        // exactly the rows l + 32c (SFB: + 128h) whose 16-byte slots its rearranged
        // words occupy, so the transpose is lane-local.  (4-byte copies straight into
        // place issue four times as many memory requests, which bounded this path.)
        const uint8_t* sa8 = reinterpret_cast<const uint8_t*>(p.sa);
        const uint8_t* sb8 = reinterpret_cast<const uint8_t*>(p.sb);
        const bool wide = (p.k & 511) == 0;
        int s = 0, prev_s = -1;
        uint32_t ph = 0, prev_ph = 0;
        auto signal = [&](int st, uint32_t sph) {
            if (!pair_warp_wait(bar_sf_raw(st), sph, abort_flag, peer_abort, p.err)) {
                aborted = true;
                return;
            }
            if (wide) {
                uint4* sfa = reinterpret_cast<uint4*>(smem + L::kOffSfa +
                                                      st * L::kKbPerStage * L::kSfaBytes);
                uint4 r[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) r[c] = sfa[c * 32 + lane];
                sfa[lane] = make_uint4(r[0].x, r[1].x, r[2].x, r[3].x);        // K block 0, word 0
                sfa[32 + lane] = make_uint4(r[0].y, r[1].y, r[2].y, r[3].y);   // K block 0, word 1
                sfa[64 + lane] = make_uint4(r[0].z, r[1].z, r[2].z, r[3].z);   // K block 1, word 0
                sfa[96 + lane] = make_uint4(r[0].w, r[1].w, r[2].w, r[3].w);   // K block 1, word 1
                uint4* sfb = reinterpret_cast<uint4*>(smem + L::kOffSfb +
                                                      st * L::kKbPerStage * L::kSfbBytes);
                // all eight rows first: the rearranged words of one half land on raw rows
                // of the other
                uint4 t[8];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int c = 0; c < 4; ++c) t[h * 4 + c] = sfb[h * 128 + c * 32 + lane];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4* u = t + h * 4;
                    // (K block, word, half) -> matrix K block * 4 + 2 word + half
                    sfb[(0 * 4 + 0 + h) * 32 + lane] = make_uint4(u[0].x, u[1].x, u[2].x, u[3].x);
                    sfb[(0 * 4 + 2 + h) * 32 + lane] = make_uint4(u[0].y, u[1].y, u[2].y, u[3].y);
                    sfb[(1 * 4 + 0 + h) * 32 + lane] = make_uint4(u[0].z, u[1].z, u[2].z, u[3].z);
                    sfb[(1 * 4 + 2 + h) * 32 + lane] = make_uint4(u[0].w, u[1].w, u[2].w, u[3].w);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(mapa_shared(bar_full(st), 0));
        };
        for (int pi = 0; !aborted; ++pi) {
            const PairPiece pc = get_piece(pi);
            if (pc.u < 0) break;
            const PairUnit w = get_unit(pc.u);
            const int64_t sa_goff = kMasked ? static_cast<int64_t>(w.g) * p.sa_g_stride : 0;
            const int64_t brow0 =
                static_cast<int64_t>(w.g) * p.n + static_cast<int64_t>(w.n_tile) * 256;
            for (int ks = pc.ks0; ks < pc.ks1 && !aborted; ++ks) {
                if (!pair_warp_wait(bar_empty(s), ph ^ 1u, abort_flag, peer_abort, p.err)) {
                    aborted = true;
                    break;
                }
                const int kb0 = ks * L::kKbPerStage;
                if (wide) {
                    // the stage's 16 bytes of every row (8 when its second K block is past K)
                    const uint32_t nbytes = kb0 + 1 < KB ? 16u : 8u;
                    const uint32_t sfa = sbase + L::kOffSfa + s * L::kKbPerStage * L::kSfaBytes;
                    const uint32_t sfb = sbase + L::kOffSfb + s * L::kKbPerStage * L::kSfbBytes;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int r = c * 32 + lane;
                        const int64_t m = static_cast<int64_t>(w.m_base) + r;
                        const bool in = m < p.rows;
                        cp_async_16(sfa + 16 * r, in ? sa8 + sa_goff + m * (p.k >> 5) + kb0 * 8 : sa8,
                                    in ? nbytes : 0u);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int nr = q * 32 + lane;
                        cp_async_16(sfb + 16 * nr, sb8 + (brow0 + nr) * (p.k >> 5) + kb0 * 8, nbytes);
                    }
                }
#pragma unroll
                for (int j = 0; j < (wide ? 0 : L::kKbPerStage); ++j) {
                    const int kb = kb0 + j;
                    const uint32_t slot = s * L::kKbPerStage + j;
                    const uint32_t sfa = sbase + L::kOffSfa + slot * L::kSfaBytes;
                    const uint32_t sfb = sbase + L::kOffSfb + slot * L::kSfbBytes;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = q * 32 + lane;
                        const int64_t m = static_cast<int64_t>(w.m_base) + r;
                        const bool in = m < p.rows && kb < KB;
                        const uint8_t* src = sa8 + sa_goff + m * (p.k >> 5) + kb * 8;
#pragma unroll
                        for (int wd = 0; wd < 2; ++wd)
                            cp_async_4(sfa + wd * 512 + lane * 16 + q * 4, in ? src + 4 * wd : sa8,
                                       in ? 4u : 0u);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int nr = q * 32 + lane;   // row of the unit's 256-row B tile
                        const bool in = kb < KB;
                        const uint8_t* src = sb8 + (brow0 + nr) * (p.k >> 5) + kb * 8;
#pragma unroll
                        for (int wd = 0; wd < 2; ++wd)
                            cp_async_4(sfb + (2 * wd + (q >> 2)) * 512 + lane * 16 + (q & 3) * 4,
                                       in ? src + 4 * wd : sb8, in ? 4u : 0u);
                    }
                }
                cp_async_mbar_arrive_noinc(bar_sf_raw(s));
                if (prev_s >= 0) signal(prev_s, prev_ph);
                prev_s = s;
                prev_ph = ph;
                if (++s == S) { s = 0; ph ^= 1u; }
            }
        }
        if (!aborted && prev_s >= 0) signal(prev_s, prev_ph);
    } else if (warp == 3) {
        // ============================================================ scale converter
        // The activation scales of every row this CTA stores, and the unit's weight
        // scales, are checked to be UE8M0 values (ue8m0_scale_ok): the conversion
        // keeps only the exponent field.  Rows that are not computed may hold anything.
        int s = 0;
        uint32_t ph = 0;
        bool bad = false;
        for (int pi = 0; !aborted; ++pi) {
            const PairPiece pc = get_piece(pi);
            if (pc.u < 0) break;
            const PairUnit w = get_unit(pc.u);
            if (p.sf_a_packed != nullptr && !kMx) {
                // packed scale images: relay the stage's arrival to the leader's full
                // barrier.  The step's four weight scales (lanes 0-3: chunk lane / 2, K
                // block lane % 2) are checked after the next arrival, one step after
                // their load was issued, so that the check never holds up a relay.
                auto load_sb = [&](int ks) {
                    const int c = lane >> 1;
                    const int kb = ks * L::kKbPerStage + (lane & 1);
                    const int nb = kSwiglu ? c * (p.n >> 8) + w.n_tile : w.n_tile * 2 + c;
                    const bool chk = lane < (w.half_n ? 2 : 4) && kb < KB;
                    return chk ? __float_as_uint(
                                     __ldg(p.sb + (static_cast<int64_t>(w.g) * p.nb_count + nb) * KB + kb))
                               : 0x3F800000u;  // 1.0: nothing to check
                };
                uint32_t sbv = load_sb(pc.ks0);
                for (int ks = pc.ks0; ks < pc.ks1; ++ks) {
                    if (!pair_warp_wait(bar_sf_raw(s), ph, abort_flag, peer_abort, p.err)) {
                        aborted = true;
                        break;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(mapa_shared(bar_full(s), 0));
                    const uint32_t cur = sbv;
                    if (ks + 1 < pc.ks1) sbv = load_sb(ks + 1);
                    bad |= !ue8m0_scale_ok(cur);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                continue;
            }
            // whether row 32 q + lane of this CTA's half is stored: the row map is loaded
            // here and first read by the checks after the piece's first arrival
            int rmap[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t m = static_cast<int64_t>(w.m_base) + q * 32 + lane;
                if constexpr (kMasked) rmap[q] = q == 0 ? __ldg(p.row_info + w.g) : 0;
                else rmap[q] = w.store && m < p.rows ? __ldg(p.row_info + m) : -1;
            }
            auto stored = [&](int q) {
                const int64_t m = static_cast<int64_t>(w.m_base) + q * 32 + lane;
                if constexpr (kMasked) return w.store && m < rmap[0] && m < p.rows;
                else return rmap[q] == w.g;
            };
            for (int ks = pc.ks0; ks < pc.ks1; ++ks) {
                if (!pair_warp_wait(bar_sf_raw(s), ph, abort_flag, peer_abort, p.err)) {
                    aborted = true;
                    break;
                }
                // raw scales of this lane's rows (32 q + lane) and of the two weight chunks
                uint32_t ra[L::kKbPerStage][4], rb[L::kKbPerStage];
                if constexpr (!kMx) {
                    const int slot0 = s * L::kKbPerStage;
#pragma unroll
                    for (int j = 0; j < L::kKbPerStage; ++j) {
                        const uint32_t* a_raw = reinterpret_cast<const uint32_t*>(
                            smem + L::kOffSaRaw + (slot0 + j) * L::kSaRawBytes);
                        const uint32_t* b_raw = reinterpret_cast<const uint32_t*>(
                            smem + L::kOffSbRaw + (slot0 + j) * L::kSbRawBytes);
#pragma unroll
                        for (int q = 0; q < 4; ++q) ra[j][q] = a_raw[32 * q + lane];
                        rb[j] = b_raw[lane & 1];
                    }
                    // One scale word per row (SFA) or column chunk (SFB) and stage: byte j
                    // is the UE8M0 scale of the stage's K block j, and the MMAs of K block j
                    // select byte j through the instruction's scale ids, so a stage needs
                    // one set of scale copies instead of one per K block.
                    auto word = [&](const uint32_t (&v)[L::kKbPerStage][4], int q) {
                        uint32_t w = 0;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            w |= ((v[j % L::kKbPerStage][q] >> 23) & 0xFFu) << (8 * j);
                        return w;
                    };
                    uint4 wv;
                    wv.x = word(ra, 0);
                    wv.y = word(ra, 1);
                    wv.z = word(ra, 2);
                    wv.w = word(ra, 3);
                    *reinterpret_cast<uint4*>(smem + L::kOffSfa + slot0 * L::kSfaBytes + 16 * lane) = wv;
                    uint32_t wb = 0;
#pragma unroll
                    for (int j = 0; j < 4; ++j) wb |= ((rb[j % L::kKbPerStage] >> 23) & 0xFFu) << (8 * j);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t v = __shfl_sync(0xffffffffu, wb, c);
                        *reinterpret_cast<uint4*>(smem + L::kOffSfb + slot0 * L::kSfbBytes + 512 * c +
                                                  16 * lane) = make_uint4(v, v, v, v);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(mapa_shared(bar_full(s), 0));
                if constexpr (!kMx) {
                    // the checks come after the arrival: they delay no stage
#pragma unroll
                    for (int j = 0; j < L::kKbPerStage; ++j) {
                        if (ks * L::kKbPerStage + j < KB) {  // zero-filled past K
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                bad |= stored(q) && !ue8m0_scale_ok(ra[j][q]);
                            // (a 128-column tile has no second weight-scale chunk)
                            bad |= lane < (w.half_n ? 1 : 2) && !ue8m0_scale_ok(rb[j]);
                        }
                    }
                }
                if (++s == S) { s = 0; ph ^= 1u; }
            }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(p.err, kErrBadScale);
    } else if (warp >= 4) {
        // ============================================================ epilogue
        const int q = warp & 3;
        const int row_in_half = q * 32 + lane;
        const uint32_t empty_leader = mapa_shared(bar_tmem_empty, 0);
        uint32_t acc_ph = 0;
        int steps_done = 0;  // pipeline steps of this CTA up to and including piece pi
        for (int pi = 0; !aborted; ++pi) {
            const PairPiece pc = get_piece(pi);
            if (pc.u < 0) break;
            steps_done += pc.ks1 - pc.ks0;
            const PairUnit w = get_unit(pc.u);
            const int64_t m = static_cast<int64_t>(w.m_base) + row_in_half;
            bool valid = w.store;
            int64_t drow;
            if constexpr (kMasked) {
                int mm = __ldg(p.row_info + w.g);
                mm = mm < 0 ? 0 : (mm > p.rows ? static_cast<int>(p.rows) : mm);
                valid = valid && m < mm;
                drow = static_cast<int64_t>(w.g) * p.rows + m;
            } else {
                drow = m;
                if (valid) {
                    const int lv = m < p.rows ? __ldg(p.row_info + m) : -1;
                    if (lv != w.g) {
                        if (lv >= p.num_groups || lv < -1) raise_error(p.err, kErrBadGroup);
                        else if (lv >= 0) raise_error(p.err, kErrMixedTile);
                        valid = false;
                    }
                }
            }
            if (!pair_warp_wait(bar_tmem_full, acc_ph, abort_flag, peer_abort, p.err)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            uint8_t* dst = reinterpret_cast<uint8_t*>(static_cast<OutT*>(p.d) + drow * p.n +
                                                      w.n_tile * 256);
            // fused gate/up: 128 code bytes of this row and its scale for the unit's block
            uint8_t* qdst = reinterpret_cast<uint8_t*>(p.d) + drow * (p.n >> 1) + w.n_tile * 128;
            float* sdst = p.q_scale + (kMasked ? static_cast<int64_t>(w.g) * p.qs_g_stride : 0) +
                          m * p.qs_row_stride + w.n_tile * p.qs_col_stride;
            if (kSwiglu && pc.kind == 0) {
                float h[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) {  // 32 gate columns and the matching up columns
                    uint32_t gv[32], uv[32];
                    tc_ld_32x32b_x32_sync(trow + 32 * c, gv);
                    tc_ld_32x32b_x32_sync(trow + 128 + 32 * c, uv);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        h[32 * c + i] = silu_f32(__uint_as_float(gv[i])) * __uint_as_float(uv[i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed_cluster(empty_leader);
                quantize_store_row(h, qdst, sdst, valid);
            } else if (pc.kind == 0) {
                // the whole 256-column row goes to registers as packed bf16/f16 pairs
                // first, so the accumulator is handed back before any global store
                uint32_t packed[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[64];
                    tc_ld_32x32b_x64_sync(trow + c * 64, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        packed[c][i] =
                            pack2<OutT>(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                }
                // all TMEM reads of this tile have completed (wait::ld); the signal
                // publishes no memory writes, so it is a relaxed arrival
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed_cluster(empty_leader);
                if (valid) {
                    const bool split = p.d_align16 != 0;
                    const int nch = w.half_n ? 2 : 4;  // 64-column chunks of the tile
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (c >= nch) break;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            st_global_32B(dst + 128 * c + 32 * i, split, packed[c][8 * i],
                                          packed[c][8 * i + 1], packed[c][8 * i + 2],
                                          packed[c][8 * i + 3], packed[c][8 * i + 4],
                                          packed[c][8 * i + 5], packed[c][8 * i + 6],
                                          packed[c][8 * i + 7]);
                        }
                    }
                }
            } else if (pc.kind == 2) {
                // tail: publish the fp32 partial of this CTA's 128 rows in slot
                // (pair, rank), laid out [32 column groups][128 rows][8 columns] so that
                // each warp store covers 1 KB of contiguous memory; each warp then
                // counts itself in the slot's ready word
                const int slot = pair_id * 2 + static_cast<int>(rank);
                float* part = p.sk_partial + static_cast<int64_t>(slot) * (128 * 256) + row_in_half * 8;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[64];
                    tc_ld_32x32b_x64_sync(trow + c * 64, v);
                    if (c == 3) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_relaxed_cluster(empty_leader);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        st_global_v8(part + (c * 8 + i) * (128 * 8), v[8 * i], v[8 * i + 1],
                                     v[8 * i + 2], v[8 * i + 3], v[8 * i + 4], v[8 * i + 5],
                                     v[8 * i + 6], v[8 * i + 7]);
                    }
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(p.sk_flags + 2 * slot, 1u);
            } else {
                // head (the pair's last piece): the A producer has staged the partial of
                // the unit's tail in the two stages after this CTA's last step, chunk c in
                // the A (c even) or B (c odd) half of stage (last + 1 + c / 2) mod S
                const int slot = (pair_id + 1) * 2 + static_cast<int>(rank);
                auto part_chunk = [&](int c) {
                    const int sc = (steps_done + (c >> 1)) % S;
                    return reinterpret_cast<const float*>(
                        smem + ((c & 1) ? L::kOffB + sc * L::kBStageBytes
                                        : L::kOffA + sc * L::kAStageBytes));
                };
                if constexpr (kSwiglu) {
                    // partial column col of this row in the staged slot: chunk col / 64,
                    // column group (col % 64) / 8, [128 rows][8 columns] per group
                    float h[128];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {  // 32 gate columns and the matching up columns
                        uint32_t gv[32], uv[32];
                        tc_ld_32x32b_x32_sync(trow + 32 * c, gv);
                        tc_ld_32x32b_x32_sync(trow + 128 + 32 * c, uv);
                        if (c == 3) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive_relaxed_cluster(empty_leader);
                        }
                        if ((c & 1) == 0) {  // gate chunk c/2 and up chunk 2 + c/2
                            if (!pair_warp_wait(bar_part(c >> 1), 0, abort_flag, peer_abort, p.err) ||
                                !pair_warp_wait(bar_part(2 + (c >> 1)), 0, abort_flag, peer_abort,
                                                p.err)) {
                                aborted = true;
                                break;
                            }
                        }
                        // gate columns 32c.. are in chunk c / 2, the up columns in chunk 2 + c / 2
                        const float* gpart = part_chunk(c >> 1) + row_in_half * 8;
                        const float* upart = part_chunk(2 + (c >> 1)) + row_in_half * 8;
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const int col = (32 * c + i) & 63;
                            const float4 gp = *reinterpret_cast<const float4*>(
                                gpart + (col >> 3) * (128 * 8) + (col & 7));
                            const float4 up = *reinterpret_cast<const float4*>(
                                upart + (col >> 3) * (128 * 8) + (col & 7));
                            h[32 * c + i] = silu_f32(__uint_as_float(gv[i]) + gp.x) *
                                            (__uint_as_float(uv[i]) + up.x);
                            h[32 * c + i + 1] = silu_f32(__uint_as_float(gv[i + 1]) + gp.y) *
                                                (__uint_as_float(uv[i + 1]) + up.y);
                            h[32 * c + i + 2] = silu_f32(__uint_as_float(gv[i + 2]) + gp.z) *
                                                (__uint_as_float(uv[i + 2]) + up.z);
                            h[32 * c + i + 3] = silu_f32(__uint_as_float(gv[i + 3]) + gp.w) *
                                                (__uint_as_float(uv[i + 3]) + up.w);
                        }
                    }
                    if (!aborted) quantize_store_row(h, qdst, sdst, valid);
                }
#pragma unroll 1
                for (int c = 0; c < (kSwiglu ? 0 : L::kPartChunks); ++c) {
                    uint32_t v[64];
                    tc_ld_32x32b_x64_sync(trow + c * 64, v);
                    if (c == 3) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_relaxed_cluster(empty_leader);
                    }
                    if (!pair_warp_wait(bar_part(c), 0, abort_flag, peer_abort, p.err)) {
                        aborted = true;
                        break;
                    }
                    // chunk c: [8 column groups][128 rows][8 columns] fp32
                    const float* part = part_chunk(c) + row_in_half * 8;
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float4 f = *reinterpret_cast<const float4*>(
                            part + (i >> 1) * (128 * 8) + 4 * (i & 1));
                        pk[2 * i] = pack2<OutT>(__uint_as_float(v[4 * i]) + f.x,
                                                __uint_as_float(v[4 * i + 1]) + f.y);
                        pk[2 * i + 1] = pack2<OutT>(__uint_as_float(v[4 * i + 2]) + f.z,
                                                    __uint_as_float(v[4 * i + 3]) + f.w);
                    }
                    if (valid && (c < 2 || !w.half_n)) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            st_global_32B(dst + 128 * c + 32 * i, p.d_align16 != 0, pk[8 * i],
                                          pk[8 * i + 1], pk[8 * i + 2], pk[8 * i + 3], pk[8 * i + 4],
                                          pk[8 * i + 5], pk[8 * i + 6], pk[8 * i + 7]);
                        }
                    }
                }
                // the slot has been copied out (all four copies completed): ready for
                // the next launch
                if (warp == 4 && lane == 0 && !aborted) p.sk_flags[2 * slot] = 0u;
                if (aborted) break;
            }
            acc_ph ^= 1u;
        }
    }

    // ---------------------------------------------------------------- teardown
    if (*abort_flag) {
        // copies issued by this CTA may still be landing in its shared memory
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 200000ull) {
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer no longer reads or signals this CTA's shared memory
    tc_fence_after();
    if (warp == 2) tmem_dealloc_pair(tmem_base, L::kTmemCols);
}

}  // namespace fp8bs
