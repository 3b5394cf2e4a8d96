/*
 * fp8bs.h -- C ABI of the GB300 (sm_103a) grouped FP8 block-scaled GEMM.
 *
 * The operation ("Adds Grouped and Batched GEMM kernels with blockscaling
 * matching DeepGEMM API", FlyDSL PR #433, section Summary):
 *
 *   D[r, n] = sum_kb  scale_a[r, kb] * scale_b[g, n/128, kb]
 *                     * sum_{k = 128*kb}^{128*kb+127} A[r, k] * B[g, n, k]
 *
 * with A and B in FP8 E4M3 (OCP "FN" encoding), one activation scale per
 * (1 row, 128 K) block and one weight scale per (128 N, 128 K) block, fp32
 * accumulation and a bf16 or f16 output rounded to nearest even.  g is the
 * group (MoE expert) of row r.  Both operands are K-major ("NT"): A row r is
 * K contiguous bytes, B[g] row n is K contiguous bytes.
 *
 * Scales are fp32 values that must be powers of two in [2^-127, 2^127]
 * (UE8M0: the page's section "DeepGEMM conformance details" rounds them with
 * ceil_to_ue8m0 and has the matrix instruction apply them).  The kernels use
 * the fp32 exponent field as the UE8M0 scale byte.  A call whose stored rows
 * read any other scale value (not a power of two, zero, negative, inf or NaN)
 * is invalid: the kernels check every scale that enters a stored row and set
 * FP8BS_DEVERR_BAD_SCALE, and the rows that read such a scale hold
 * undefined values.  Scales of rows that are not computed are not read for
 * any result and are not checked.  For classic fp32 scales (amax / 448) use
 * the *_fp32_scales entry points.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major and
 *    contiguous unless a leading dimension says otherwise.  The library keeps
 *    none of them past the call except as a key of its tensor-map cache.
 *  - A, B and D must be 16-byte aligned; scale tensors 4-byte aligned (16-byte
 *    for the transposed activation-scale layout, whose ld_sa must be a
 *    multiple of 4).  N and K must be positive multiples of 128.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous: they validate, enqueue one kernel and return.  The kernel
 *    is launched with programmatic stream serialization: its CTAs may be
 *    scheduled while the preceding kernel on the stream is still finishing,
 *    but each executes griddepcontrol.wait before it reads or writes device
 *    memory, so stream order is kept.  Each kernel also signals
 *    griddepcontrol.launch_dependents early, which lets a following kernel
 *    launched the same way start on the SMs this one has freed.
 *  - Scratch: the CTA-pair kernel balances its last rounds with a stream-K
 *    split whose fp32 partial tiles live in a per-(device, stream) workspace
 *    (about 20 MB on a 152-SM GB300) that the library allocates with
 *    cudaMalloc on the first such call on that stream and keeps until exit.
 *    If that first call happens while the stream is being captured into a
 *    CUDA graph, or the allocation fails, the call runs without the split
 *    (same results, less balanced).  Calls can be captured into CUDA graphs;
 *    a capture on a stream that has already run one call replays to the same
 *    bits as the eager call.  Launches on one stream share the
 *    workspace safely; concurrent launches on different streams use
 *    different workspaces.  The contiguous variants keep their list of
 *    expert tile pairs in shared memory up to 524288 rows (507904 for MXFP4)
 *    and above that in a second per-stream workspace (about 4 bytes per
 *    128-row tile per SM, up to 4194304 rows), allocated the same way; when
 *    it cannot be had, gemm_grouped_contiguous runs the one-CTA kernel
 *    instead (same results) and the other contiguous entry points return
 *    FP8BS_ERR_CUDA.
 *  - Scale images: with row-major activation scales (sa_layout FP8BS_SA_MK
 *    and k > 128), gemm_grouped_contiguous, gemm_grouped_masked and the two
 *    *_silu_mul_quant entry points launch a short kernel before the GEMM that
 *    writes the call's scales as the UE8M0 bytes the tensor core reads, in a
 *    third per-stream workspace of (128-row tiles + num_groups * n/128) *
 *    ceil(k/256) * 512 bytes, allocated the same way.  When it cannot be had
 *    the GEMM converts the fp32 scales itself (same results).
 *  - A per-stream workspace is allocated at twice the size its call needs; a
 *    larger call that outgrows it replaces it by one at least twice its size,
 *    and the old buffer is kept, not freed, until exit, so a CUDA graph
 *    captured while it was current stays valid.  A graph keeps
 *    using the workspaces of the stream it was captured on: do not replay it
 *    on another stream while calls run on that one.
 *  - Kernels: gemm_grouped_contiguous and gemm_grouped_masked run a CTA-pair
 *    kernel (256 x 256 output tiles on two SMs) for every n; when n % 256 == 128
 *    the last column tile is 128 wide.  D may be 16-byte aligned (32-byte
 *    stores when it is 32-byte aligned, 16-byte stores otherwise).
 *  - Rows that are not computed (grouped_layout == -1, or m >= masked_m[g])
 *    are not written: D keeps its prior contents there.
 *  - Return value: FP8BS_OK, or an error code; nothing is enqueued on error.
 *    Device-side problems (masked_m out of range, a 128-row tile holding two
 *    experts, a scale that is not a UE8M0 value, a pipeline wait that exceeded
 *    its time limit) are recorded in a per-device error word read by
 *    fp8bs_device_error().
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum fp8bs_status {
    FP8BS_OK = 0,
    FP8BS_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment, layout or dtype code */
    FP8BS_ERR_UNSUPPORTED = 2, /* device is not compute capability 10.x / sm_103 family */
    FP8BS_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    FP8BS_ERR_DEVICE = 4       /* fp8bs_device_error(): the device error word was set */
};

enum fp8bs_out_dtype { FP8BS_OUT_BF16 = 0, FP8BS_OUT_F16 = 1 };

/* Activation-scale layouts (page section Summary: "including the transposed
 * [scale_k, M] activation-scale layout"). */
enum fp8bs_sa_layout {
    FP8BS_SA_MK = 0, /* [rows, K/128] row-major (per group [M_max, K/128] when masked) */
    FP8BS_SA_KM = 1  /* transposed [K/128, ld_sa] (per group [K/128, ld_sa] when masked) */
};

/* Device error word bits (fp8bs_device_error). */
#define FP8BS_DEVERR_TIMEOUT 0x1u       /* a pipeline wait gave up; the kernel exited early */
#define FP8BS_DEVERR_MASKED_M 0x2u      /* masked_m[g] < 0 or > M_max (clamped) */
#define FP8BS_DEVERR_MIXED_TILE 0x4u    /* a 128-row tile held rows of two experts */
#define FP8BS_DEVERR_BAD_GROUP 0x8u     /* grouped_layout value >= num_groups or < -1 */
#define FP8BS_DEVERR_BAD_SCALE 0x10u    /* an E4M3-path scale of a stored row (or of its
                                           weight block) is not a power of two in
                                           [2^-127, 2^127] */

/*
 * Contiguous grouped GEMM (DeepGEMM's m_grouped_fp8_gemm_nt_contiguous
 * contract, page section Summary).
 *
 *   a               E4M3 [m_sum, k]
 *   scale_a         fp32, sa_layout FP8BS_SA_MK: [m_sum, k/128];
 *                   FP8BS_SA_KM: [k/128, ld_sa] with ld_sa >= m_sum, ld_sa % 4 == 0
 *   ld_sa           leading dimension of the KM layout (ignored for MK)
 *   b               E4M3 [num_groups, n, k]
 *   scale_b         fp32 [num_groups, n/128, k/128]
 *   grouped_layout  int32 [m_sum]: the group of each row, -1 for a padding row.
 *                   Experts are padded to multiples of 128 rows: the first
 *                   row of each aligned 128-row tile names the tile's group
 *                   (-1 there skips the whole tile).  Rows of another group
 *                   inside a tile are left unwritten and set
 *                   FP8BS_DEVERR_MIXED_TILE; ids outside [-1, num_groups) set
 *                   FP8BS_DEVERR_BAD_GROUP.
 *   d               out_dtype [m_sum, n]
 *   m_sum >= 0 (0 is a no-op), n, k > 0 multiples of 128, num_groups >= 1.
 */
int gemm_grouped_contiguous(const void* a, const float* scale_a, int sa_layout, int64_t ld_sa,
                            const void* b, const float* scale_b, const int32_t* grouped_layout,
                            void* d, int out_dtype, int64_t m_sum, int64_t n, int64_t k,
                            int64_t num_groups, void* stream);

/*
 * Masked grouped GEMM (DeepGEMM's m_grouped_fp8_gemm_nt_masked contract, page
 * section Summary): group g computes only its first masked_m[g] rows.
 *
 *   a          E4M3 [num_groups, m_max, k]
 *   scale_a    fp32, FP8BS_SA_MK: [num_groups, m_max, k/128];
 *              FP8BS_SA_KM: [num_groups, k/128, ld_sa], ld_sa >= m_max, ld_sa % 4 == 0
 *   b, scale_b as for the contiguous variant
 *   masked_m   int32 [num_groups] in DEVICE memory, 0 <= masked_m[g] <= m_max
 *              (values outside are clamped and flagged FP8BS_DEVERR_MASKED_M)
 *   expected_m a hint of the typical masked_m; it never changes results (may be 0)
 *   d          out_dtype [num_groups, m_max, n]
 *   1 <= num_groups <= 1024 (the kernels keep a prefix over the groups in shared
 *   memory; FP8BS_ERR_INVALID_ARG above), m_max >= 0, n and k as for the
 *   contiguous variant.
 */
int gemm_grouped_masked(const void* a, const float* scale_a, int sa_layout, int64_t ld_sa,
                        const void* b, const float* scale_b, const int32_t* masked_m,
                        int64_t expected_m, void* d, int out_dtype, int64_t num_groups,
                        int64_t m_max, int64_t n, int64_t k, void* stream);

/*
 * Fused first MoE GEMM: the grouped GEMM of the gate/up projection followed by
 * SiLU(gate) * up and requantisation for the down projection.
 *   - silu_mul of the gate and up halves: "flydsl mxfp4 a4w4 MoE: bring
 *     gemm1/gemm2 to parity with the HIP backend" (aiter PR #3828), section
 *     gemm1 (the exponential is the hardware one, __expf);
 *   - the quantiser of the activations of "Adds Grouped and Batched GEMM
 *     kernels with blockscaling matching DeepGEMM API", DeepGEMM conformance
 *     details: per (1,128) block, scale = smallest power of two >= amax / 448
 *     (amax at least 1e-4), codes = E4M3 round-to-nearest-even of h / scale.
 *
 * For each computed row r of expert g and output column j < n/2:
 *     gate = acc(r, j), up = acc(r, n/2 + j), with acc the block-scaled product
 *            of gemm_grouped_contiguous against B[g] (rows [0, n/2) of each
 *            expert's B are the gate projection, rows [n/2, n) the up one);
 *     h    = gate / (1 + exp(-gate)) * up, in fp32;
 *     out[r, j] = E4M3(h / out_scale[r, j/128]).
 * The scale exponent and the codes are decided in fp32 from the fp32
 * accumulator, so a code whose exact value lies within a few fp32 ulps of an
 * E4M3 rounding boundary (or a scale whose amax / 448 lies that close to a
 * power of two) may come out as either neighbour.
 *
 *   a, scale_a, sa_layout, ld_sa, b, scale_b, grouped_layout: as for
 *              gemm_grouped_contiguous, with n = 2 * (output columns)
 *   out        E4M3 [m_sum, n/2], 32-byte aligned
 *   out_scale  fp32, out_scale_layout FP8BS_SA_MK: [m_sum, n/256];
 *              FP8BS_SA_KM: [n/256, ld_out_scale], ld_out_scale >= m_sum,
 *              ld_out_scale % 4 == 0, 16-byte aligned.  Either is a scale_a
 *              layout of gemm_grouped_contiguous, so (out, out_scale) is the
 *              activation operand of the down projection as it stands.
 *   n % 256 == 0 (n/2 a multiple of 128), m_sum <= 4194304, num_groups < 2^15:
 *              the op runs on the CTA-pair kernel only; other shapes return
 *              FP8BS_ERR_INVALID_ARG.  Above 524288 rows the pair list lives in
 *              a per-stream device workspace (grown on first use, like the
 *              stream-K scratch): a call that would need to grow it while the
 *              stream is being captured returns FP8BS_ERR_CUDA.
 * Rows with grouped_layout == -1 are written neither in out nor in out_scale.
 * Scratch as for gemm_grouped_contiguous (the per-stream stream-K workspace).
 */
int gemm_grouped_contiguous_silu_mul_quant(const void* a, const float* scale_a, int sa_layout,
                                           int64_t ld_sa, const void* b, const float* scale_b,
                                           const int32_t* grouped_layout, void* out,
                                           float* out_scale, int out_scale_layout,
                                           int64_t ld_out_scale, int64_t m_sum, int64_t n,
                                           int64_t k, int64_t num_groups, void* stream);

/*
 * Masked variant of gemm_grouped_contiguous_silu_mul_quant (the decode-time
 * layout of gemm_grouped_masked): group g computes its first masked_m[g] rows.
 *   out        E4M3 [num_groups, m_max, n/2], 32-byte aligned
 *   out_scale  fp32, FP8BS_SA_MK: [num_groups, m_max, n/256];
 *              FP8BS_SA_KM: [num_groups, n/256, ld_out_scale],
 *              ld_out_scale >= m_max, ld_out_scale % 4 == 0, 16-byte aligned
 *   other arguments as for gemm_grouped_masked, with n % 256 == 0.
 * Rows m >= masked_m[g] are written neither in out nor in out_scale.
 */
int gemm_grouped_masked_silu_mul_quant(const void* a, const float* scale_a, int sa_layout,
                                       int64_t ld_sa, const void* b, const float* scale_b,
                                       const int32_t* masked_m, int64_t expected_m, void* out,
                                       float* out_scale, int out_scale_layout,
                                       int64_t ld_out_scale, int64_t num_groups, int64_t m_max,
                                       int64_t n, int64_t k, void* stream);

/*
 * Grouped GEMM with arbitrary fp32 block scales (software promotion).
 *
 * Same arguments, layouts and results contract as gemm_grouped_contiguous /
 * gemm_grouped_masked, but scale_a and scale_b may hold any finite fp32
 * values, not only the powers of two the tensor core applies itself: the
 * product of each 128-K block is formed without scales (tcgen05.mma
 * kind::f8f6f4), then multiplied by sa[r, kb] * sb[g, n/128, kb] (rounded to
 * fp32) and added in fp32 by the CUDA cores -- the promotion scheme of the
 * DeepGEMM path the "Adds Grouped and Batched GEMM kernels with blockscaling
 * matching DeepGEMM API" page (DeepGEMM conformance details) describes for
 * hardware without scaled matrix instructions.  Also an independent check of
 * the hardware-scaled path on power-of-two scales.
 *
 * Runs on the CTA-pair kernel only: n % 256 == 0, d 32-byte aligned, and for
 * the contiguous variant m_sum <= 4194304 rows and num_groups < 2^15; other
 * shapes return FP8BS_ERR_INVALID_ARG.  No stream-K tail.  Above 524288 rows
 * the pair list lives in the per-stream device workspace, as for
 * gemm_grouped_contiguous_silu_mul_quant (FP8BS_ERR_CUDA when it would have
 * to grow during stream capture); below that no scratch memory is used.
 */
int gemm_grouped_contiguous_fp32_scales(const void* a, const float* scale_a, int sa_layout,
                                        int64_t ld_sa, const void* b, const float* scale_b,
                                        const int32_t* grouped_layout, void* d, int out_dtype,
                                        int64_t m_sum, int64_t n, int64_t k, int64_t num_groups,
                                        void* stream);

int gemm_grouped_masked_fp32_scales(const void* a, const float* scale_a, int sa_layout,
                                    int64_t ld_sa, const void* b, const float* scale_b,
                                    const int32_t* masked_m, int64_t expected_m, void* d,
                                    int out_dtype, int64_t num_groups, int64_t m_max, int64_t n,
                                    int64_t k, void* stream);

/*
 * MXFP4 (a4w4) grouped GEMM: both operands in the OCP Microscaling FP4
 * format -- E2M1 elements (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) with one
 * E8M0 scale byte 2^(e - 127) per 32 consecutive elements along K -- the MoE
 * GEMM format of "flydsl mxfp4 a4w4 MoE: bring gemm1/gemm2 to parity with the
 * HIP backend" (Summary).  D[r, n] = sum over 32-element blocks j of
 * 2^(sa[r,j]-127) * 2^(sb[g,n,j]-127) * sum_{k in j} A[r,k] * B[g,n,k], fp32
 * accumulation (tcgen05.mma kind::mxf4, scales applied by the tensor core).
 *
 *   a        packed E2M1 [m_sum, k/2] (contiguous) or [num_groups, m_max, k/2]
 *            (masked); element 2i in the low nibble of byte i; 16-byte aligned
 *   scale_a  E8M0 bytes [m_sum, k/32] or [num_groups, m_max, k/32]; 4-byte aligned
 *   b        packed E2M1 [num_groups, n, k/2], 16-byte aligned
 *   scale_b  E8M0 bytes [num_groups, n, k/32] (one per row of B and 32-element
 *            block), 4-byte aligned
 *   d        out_dtype [m_sum, n] or [num_groups, m_max, n], 32-byte aligned
 *   n % 256 == 0, k % 256 == 0; contiguous: m_sum <= 4194304 rows, num_groups
 *   < 2^15 (above 507904 rows the pair list lives in the per-stream device
 *   workspace, FP8BS_ERR_CUDA if it would have to grow during stream capture);
 *   masked: num_groups <= 1024.
 *   grouped_layout / masked_m / expected_m as for the E4M3 variants.
 * Runs on the CTA-pair kernel (with the stream-K tail for the contiguous
 * variant).
 */
int gemm_grouped_contiguous_mxfp4(const void* a, const uint8_t* scale_a, const void* b,
                                  const uint8_t* scale_b, const int32_t* grouped_layout, void* d,
                                  int out_dtype, int64_t m_sum, int64_t n, int64_t k,
                                  int64_t num_groups, void* stream);

int gemm_grouped_masked_mxfp4(const void* a, const uint8_t* scale_a, const void* b,
                              const uint8_t* scale_b, const int32_t* masked_m, int64_t expected_m,
                              void* d, int out_dtype, int64_t num_groups, int64_t m_max,
                              int64_t n, int64_t k, void* stream);

/*
 * Contiguous grouped GEMM that allocates no device memory.  (No counterpart on
 * the pages: an addition for callers that may not call cudaMalloc -- for
 * example code that runs under a memory pool or allocator that owns all device
 * memory, inside an allocation-free inference runtime, or while another
 * component forbids allocations on the device.)
 *
 * Same arguments and results as gemm_grouped_contiguous.  It runs the CTA-pair
 * kernel, whose stream-K scratch (fp32 partial tiles and their slot counters)
 * lives in a statically sized device array of this library instead of a
 * cudaMalloc'd workspace:
 *  - size: 160 slots of 128 x 256 fp32 (2 per CTA pair, up to 80 pairs) plus
 *    1280 bytes of counters, about 20 MiB; every GPU that loads the library
 *    holds it until the process exits.  A device that fits more than 80 CTA
 *    pairs runs this entry point on 80 of them (same results);
 *  - the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current;
 *  - every call clears the slot counters (cudaMemsetAsync on `stream`) and
 *    then launches, so unlike the other entry points its kernel does not
 *    start early on SMs freed by the preceding kernel on the stream; calls
 *    share the array, so calls that overlap on the GPU (for instance on two
 *    streams at once) race and give wrong results;
 *  - no cudaMalloc, cudaFree or other allocating routine is called, and the
 *    TMA tensor maps are encoded on the stack for every call.
 * Returns FP8BS_ERR_INVALID_ARG, in addition to the cases of
 * gemm_grouped_contiguous, for shapes the CTA-pair kernel does not take
 * (m_sum > 524288 rows, num_groups >= 2^15).
 */
int gemm_grouped_contiguous_noalloc(const void* a, const float* scale_a, int sa_layout,
                                    int64_t ld_sa, const void* b, const float* scale_b,
                                    const int32_t* grouped_layout, void* d, int out_dtype,
                                    int64_t m_sum, int64_t n, int64_t k, int64_t num_groups,
                                    void* stream);

/* Synchronises `device`, returns the FP8BS_DEVERR_* bits recorded since the
 * last call in *flags and clears them.  Returns FP8BS_ERR_DEVICE when any bit
 * was set, FP8BS_OK otherwise (or FP8BS_ERR_CUDA / _INVALID_ARG). */
int fp8bs_device_error(int device, uint32_t* flags);

/* Static description of an error code (never NULL). */
const char* fp8bs_status_string(int status);

/* Drops every cached TMA tensor map (host memory only).  Call after freeing
 * tensors whose addresses may be reused with other shapes; the cache key
 * includes address, shape and strides, so stale entries are never wrong,
 * only kept. */
int fp8bs_clear_cache(void);

/* Test hook for the failure path (0 = off, the default).  FP8BS_DEBUG_STALL_MMA
 * makes every later launch of the CTA-pair kernel wait, in its MMA thread, on
 * a barrier nothing arrives on: the wait gives up after its time limit (4 s),
 * the launch aborts (both CTAs of every pair stop, let their copies land,
 * free tensor memory and exit) and FP8BS_DEVERR_TIMEOUT is recorded.  D is
 * then undefined.  Returns FP8BS_ERR_INVALID_ARG for unknown bits. */
#define FP8BS_DEBUG_STALL_MMA 0x1u
/* FP8BS_DEBUG_SINGLE_CTA routes later gemm_grouped_contiguous and
 * gemm_grouped_masked calls to the single-CTA kernel (128-row tiles), which
 * otherwise runs only when the contiguous pair list cannot be had: a
 * cross-check of the two kernels on the same problem.  Results are within
 * the same tolerances; nothing else changes. */
#define FP8BS_DEBUG_SINGLE_CTA 0x2u
int fp8bs_set_debug_flags(uint32_t flags);

/* Library ABI version (1). */
int fp8bs_abi_version(void);

/* Number of kernels this library has launched in this process, over all
 * devices and streams: a host-side counter, raised by one for each kernel
 * launch the CUDA runtime accepted (the scale pre-pass and the GEMM of a call
 * are two; the counter-clearing cudaMemsetAsync of
 * gemm_grouped_contiguous_noalloc is not a kernel of the library and does not
 * count).  A launch captured into a CUDA graph counts once, when captured, not
 * at each replay.  Never fails. */
uint64_t fp8bs_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
