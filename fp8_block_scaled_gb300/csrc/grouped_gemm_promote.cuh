// Grouped FP8 GEMM with software promotion of the block scales.
//
// Same operation and layouts as the block-scaled kernels ("Adds Grouped and
// Batched GEMM kernels with blockscaling matching DeepGEMM API", FlyDSL PR
// #433, section Summary), but the scales may be any fp32 values, not only the
// powers of two the tensor core applies itself (the same page, DeepGEMM
// conformance details: the MI300 path promotes in software):
//
//   D[r, n] = sum_kb  (sa[r, kb] * sb[g, n/128, kb]) * P_kb[r, n],
//   P_kb[r, n] = sum_{k in block kb} A[r, k] * B[g, n, k]
//
// Each 128-K block's unscaled product P_kb comes from four tcgen05.mma
// kind::f8f6f4 (E4M3 x E4M3, fp32) into one of two 256-column tensor-memory
// buffers, so the MMAs of block kb+1 run while block kb is promoted.  Eight
// promotion warps read P_kb, multiply it by the block's fp32 scale product and
// add it to accumulators held in registers: warp 4 + 4h + q owns TMEM lane
// quarter q (rows 32q..32q+31 of the CTA's 128) and columns 128h..128h+127,
// one row per thread, 128 fp32 accumulators per thread.
//
// CTA pair as in grouped_gemm_pair.cuh (256 x 256 units, cta_group::2 MMAs,
// A/B staging, pair-list scheduling), round-robin units without the stream-K
// tail.  Warp roles per CTA:
//   warp 0   A producer (TMA; the leader arms the full barrier for both CTAs)
//   warp 2   B producer (after allocating the pair's tensor memory)
//   warp 1   leader only, one thread: tcgen05.mma issue, commits multicast
//   warp 3   idle (no scale staging: the promotion warps read the scales)
//   warps 4-11  promotion and epilogue
#pragma once

#include "grouped_gemm_pair.cuh"

namespace fp8bs {

constexpr int kPromoteThreads = 384;

struct PromoteLayout {
    static constexpr int kKbPerStage = 2;
    static constexpr int kStages = 3;
    static constexpr int kTileBytes = 128 * kBK;
    static constexpr int kAStageBytes = kKbPerStage * kTileBytes;
    static constexpr int kBStageBytes = kKbPerStage * kTileBytes;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kAStageBytes;
    static constexpr int kOffBar = kOffB + kStages * kBStageBytes;
    // full[S], empty[S], p_full[2], p_empty[2], drain
    static constexpr int kNumBars = 2 * kStages + 5;
    static constexpr int kPrefetchStages = 3;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // slot, abort, scan scratch
    static constexpr int kMiscBytes = 16 + 2 * kMaxScanWarps * 4;
    static constexpr int kOffList = (kOffMisc + kMiscBytes + 15) / 16 * 16;
    static constexpr int kListEntries = kPairMaxTiles + 1;
    static constexpr int kBytes = kOffList + kListEntries * 4;
    static constexpr int kAlignSlack = 1024;
    static constexpr int kTmemCols = 512;                     // two 256-column partial buffers
    static_assert(kBytes + kAlignSlack <= 232448, "shared memory budget");
    static_assert(kPairMaxTiles * 4 <= kStages * kAStageBytes, "prologue scratch");
    static_assert(kPairMaxTilesWs * 4 <= kStages * (kAStageBytes + kBStageBytes) &&
                      kOffB == kOffA + kStages * kAStageBytes,
                  "prologue scratch of a workspace-sized list (A and B stages contiguous)");
};

// tcgen05 instruction descriptor, kind::f8f6f4: fp32 accumulator (bits 4-5 = 1),
// E4M3 A and B (format 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc_f8(int m, int n) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

template <typename OutT, bool kMasked>
__global__ void __launch_bounds__(kPromoteThreads, 1)
grouped_gemm_promote_kernel(const __grid_constant__ CUtensorMap tmap_a,
                            const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
    using L = PromoteLayout;
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
    auto bar_p_full = [&](int b) { return sbase + L::kOffBar + 8u * (2 * S + b); };
    auto bar_p_empty = [&](int b) { return sbase + L::kOffBar + 8u * (2 * S + 2 + b); };
    const uint32_t bar_drain = sbase + L::kOffBar + 8u * (2 * S + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
    int* scan_scratch = reinterpret_cast<int*>(smem + L::kOffMisc + 16);
    // The pair list's address is formed again at every use instead of being held
    // in a register for the whole kernel: a live 64-bit pointer here made the
    // promotion warps spill.
    auto list = [&]() {
        if (p.list_ws == nullptr) return reinterpret_cast<int*>(smem + L::kOffList);
        return p.list_ws + static_cast<int64_t>(cta_index_x()) * p.list_ws_stride;
    };
    const uint32_t peer_abort = mapa_shared(smem_addr(smem + L::kOffMisc + 4), rank ^ 1u);

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full(s), 2);       // leader's A and B producers (expect_tx for both CTAs)
            mbar_init(bar_empty(s), 1);      // leader's multicast commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_p_full(b), 1);     // leader's multicast commit
            mbar_init(bar_p_empty(b), 16);   // 8 promotion warps x 2 CTAs
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
    }
    // inputs, outputs and the error word may belong to the grid this launch follows
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp == 2) {
        tmem_alloc_pair(smem_addr(tmem_slot), L::kTmemCols);
        tmem_relinquish_pair();
    }
    const int total_units =
        build_units<kMasked, kPromoteThreads>(p, smem + L::kOffA, list(), scan_scratch);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // peer barriers initialised, tensor memory allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    auto get_unit = [&](int u) { return unit_of<kMasked>(p, list(), total_units, u, rank); };

    constexpr uint32_t kIdesc = make_idesc_f8(2 * kBM, 256);
    const int KB = p.kb_count;
    const int NKS = (KB + L::kKbPerStage - 1) / L::kKbPerStage;
    bool aborted = false;

    if (warp == 0 || warp == 2) {
        // ============================================================ producers
        const bool is_a = warp == 0;
        const CUtensorMap* map = is_a ? &tmap_a : &tmap_b;
        const uint32_t op_off = is_a ? L::kOffA : L::kOffB;
        int s = 0;
        uint32_t ph = 0;
        for (int u = pair_id; u < total_units && !aborted; u += num_pairs) {
            const PairUnit w = get_unit(u);
            const int32_t row0 =
                is_a ? static_cast<int32_t>(kMasked ? static_cast<int64_t>(w.g) * p.rows + w.m_base
                                                    : static_cast<int64_t>(w.m_base))
                     : w.g * p.n + w.n_tile * 256 + static_cast<int>(rank) * 128;
            const bool pf_owner = prefetch_owner_of<kMasked>(p, total_units, u, is_a);
            for (int ks = 0; ks < NKS; ++ks) {
                if (!pair_warp_wait(bar_empty(s), ph ^ 1u, abort_flag, peer_abort, p.err)) {
                    aborted = true;
                    break;
                }
                if (lane == 0) {
                    if (leader) mbar_arrive_expect_tx(bar_full(s), 2u * L::kAStageBytes);
                    tma_load_3d_pair(sbase + op_off + s * L::kAStageBytes, map, 0, row0,
                                     ks * L::kKbPerStage, mapa_shared(bar_full(s), 0));
                    // warm L2 with the box of this unit kPrefetchStages steps later (one
                    // prefetcher per shared tile, as in the pair kernel)
                    if (pf_owner && ks + L::kPrefetchStages < NKS)
                        tma_prefetch_3d(map, 0, row0, (ks + L::kPrefetchStages) * L::kKbPerStage);
                }
                if (++s == S) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer (leader)
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t kc = 0;  // K blocks issued so far: partial buffer kc & 1, use kc >> 1
            bool issued_any = false;
            for (int u = pair_id; u < total_units && !aborted; u += num_pairs) {
                for (int ks = 0; ks < NKS && !aborted; ++ks) {
                    if (!pair_wait(bar_full(s), ph, abort_flag, peer_abort, p.err)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < L::kKbPerStage; ++j) {
                        const int kb = ks * L::kKbPerStage + j;
                        if (kb >= KB) break;
                        const uint32_t b = kc & 1u;
                        if (!pair_wait(bar_p_empty(b), ((kc >> 1) & 1u) ^ 1u, abort_flag,
                                       peer_abort, p.err)) {
                            aborted = true;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = make_desc_sw128(sbase + L::kOffA + s * L::kAStageBytes +
                                                               j * L::kTileBytes);
                        const uint64_t bdesc = make_desc_sw128(sbase + L::kOffB + s * L::kBStageBytes +
                                                               j * L::kTileBytes);
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k)
                            tc_mma_pair_f8(tmem_base + 256u * b, adesc + 2u * k, bdesc + 2u * k,
                                           kIdesc, k > 0 ? 1u : 0u);
                        tc_commit_pair_mc(bar_p_full(b), 0x3);
                        issued_any = true;
                        ++kc;
                    }
                    if (aborted) break;
                    tc_commit_pair_mc(bar_empty(s), 0x3);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            if (aborted && issued_any) {
                tc_commit_pair_mc(bar_drain, 0x1);
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar_drain, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ============================================================ promotion + epilogue
        const int q = warp & 3;
        const int half = (warp - 4) >> 2;  // column half of the 256-column unit
        const int row_in_half = q * 32 + lane;
        const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + 128u * half;
        uint32_t kc = 0;
        for (int u = pair_id; u < total_units && !aborted; u += num_pairs) {
            const PairUnit w = get_unit(u);
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
            // this row's activation scales and the unit's 128-column weight-scale chunk
            const bool row_in = m < p.rows;
            const float* sa_row = p.sa + (kMasked ? static_cast<int64_t>(w.g) * p.sa_g_stride : 0) +
                                  (row_in ? m : 0) * p.sa_row_stride;
            const float* sb_blk =
                p.sb + (static_cast<int64_t>(w.g) * p.nb_count + w.n_tile * 2 + half) * KB;
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
            // the scales of K block kb + 4 are fetched while block kb is promoted (a
            // global load takes longer than one block's promotion)
            auto sa_at = [&](int kb) { return kb < KB ? __ldg(sa_row + kb * p.sa_kb_stride) : 0.0f; };
            auto sb_at = [&](int kb) { return kb < KB ? __ldg(sb_blk + kb) : 0.0f; };
            float a0 = sa_at(0), a1 = sa_at(1), a2 = sa_at(2), a3 = sa_at(3);
            float b0 = sb_at(0), b1 = sb_at(1), b2 = sb_at(2), b3 = sb_at(3);
            for (int kb = 0; kb < KB; ++kb) {
                const float scale = a0 * b0;
                a0 = a1; a1 = a2; a2 = a3; a3 = sa_at(kb + 4);
                b0 = b1; b1 = b2; b2 = b3; b3 = sb_at(kb + 4);
                const uint32_t b = kc & 1u;
                if (!pair_warp_wait(bar_p_full(b), (kc >> 1) & 1u, abort_flag, peer_abort,
                                    p.err)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[16];
                    tc_ld_32x32b_x16_sync(trow + 256u * b + 16 * c, v);
#pragma unroll
                    for (int i = 0; i < 16; i += 2)
                        fma2_scaled(acc[16 * c + i], acc[16 * c + i + 1], v[i], v[i + 1], scale);
                }
                // all reads of the buffer have completed (wait::ld): hand it back
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed_cluster(mapa_shared(bar_p_empty(b), 0));
                ++kc;
            }
            if (aborted) break;
            if (valid) {
                uint8_t* dst = reinterpret_cast<uint8_t*>(static_cast<OutT*>(p.d) + drow * p.n +
                                                          w.n_tile * 256 + half * 128);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    st_global_v8(dst + 32 * i, pack2<OutT>(acc[16 * i], acc[16 * i + 1]),
                                 pack2<OutT>(acc[16 * i + 2], acc[16 * i + 3]),
                                 pack2<OutT>(acc[16 * i + 4], acc[16 * i + 5]),
                                 pack2<OutT>(acc[16 * i + 6], acc[16 * i + 7]),
                                 pack2<OutT>(acc[16 * i + 8], acc[16 * i + 9]),
                                 pack2<OutT>(acc[16 * i + 10], acc[16 * i + 11]),
                                 pack2<OutT>(acc[16 * i + 12], acc[16 * i + 13]),
                                 pack2<OutT>(acc[16 * i + 14], acc[16 * i + 15]));
            }
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
