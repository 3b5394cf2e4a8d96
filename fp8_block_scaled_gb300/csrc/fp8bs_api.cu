// C ABI of the grouped FP8 block-scaled GEMM (declared in include/fp8bs.h):
// argument validation, the TMA tensor-map cache, per-device state and the
// kernel launches.  The operation and its two variants are those of the page
// "Adds Grouped and Batched GEMM kernels with blockscaling matching DeepGEMM
// API" (FlyDSL PR #433), section Summary; the raw-pointer argument style
// follows "flydsl mxfp4 a4w4 MoE: bring gemm1/gemm2 to parity with the HIP
// backend" (aiter PR #3828), section Changes / ABI.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "fp8bs.h"
#include "grouped_gemm.cuh"
#include "grouped_gemm_pair.cuh"
#include "grouped_gemm_promote.cuh"
#include "scale_pack.cuh"

// Per-device error word written by the kernels (FP8BS_DEVERR_* bits).
__device__ uint32_t g_fp8bs_error_word;

namespace {

using fp8bs::GemmParams;
using fp8bs::SmemLayout;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int status = FP8BS_OK;      // FP8BS_ERR_UNSUPPORTED when the device is not sm_103
    int sms = 0;
    uint32_t* err = nullptr;    // device address of g_fp8bs_error_word
    bool attr_set[32] = {};
    int max_clusters[32] = {};  // co-resident CTA pairs of each pair-kernel instantiation
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_launches{0};  // kernels launched (fp8bs_kernel_launches)
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct MapKey {
    int dev;
    const void* ptr;
    uint64_t inner, outer, box_outer, box_kb;  // box_kb = 0: 2-D map
    bool operator<(const MapKey& o) const {
        return std::tie(dev, ptr, inner, outer, box_outer, box_kb) <
               std::tie(o.dev, o.ptr, o.inner, o.outer, o.box_outer, o.box_kb);
    }
};
std::map<MapKey, CUtensorMap> g_maps;

// Stream-K scratch of the CTA-pair kernel, one per (device, stream): launches on
// one stream run one after another, so they may share it; launches on different
// streams may overlap and must not.
struct SkWorkspace {
    float* partial = nullptr;
    uint32_t* flags = nullptr;
    int slots = 0;
};
// Buffers of the per-stream workspaces below that a larger call replaced.  They are
// kept, not freed, until the process exits: a CUDA graph captured while one of them
// was current still points at it.  The pair list and the scale images are allocated
// at twice the size their call needs and grow to at least twice their size, so calls
// of varying sizes (the row count of a MoE layer changes with every batch) seldom
// allocate, and the kept buffers add up to less than the current ones.
std::vector<void*> g_retired;

// cudaMalloc with this thread's stream-capture mode relaxed for the call.  Callers
// never allocate while the call's own stream is capturing; a capture in global mode
// on another stream (torch's default) would otherwise make the allocation fail and
// invalidate that capture.
cudaError_t malloc_outside_capture(void** ptr, size_t bytes) {
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    const cudaError_t e = cudaMalloc(ptr, bytes);
    cudaThreadExchangeStreamCaptureMode(&mode);
    return e;
}

std::map<std::pair<int, void*>, SkWorkspace> g_sk;
constexpr size_t kSkSlotBytes = 128 * 256 * sizeof(float);

// Returns the stream's workspace with at least `slots` slots, allocating it on
// first use; nullptr (stream-K off for this launch) when that would need an
// allocation while the stream is being captured, or when allocation fails.
SkWorkspace* sk_workspace(int dev, cudaStream_t stream, int slots) {
    auto key = std::make_pair(dev, static_cast<void*>(stream));
    auto it = g_sk.find(key);
    if (it != g_sk.end() && it->second.slots >= slots) return &it->second;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return nullptr;
    }
    SkWorkspace w;
    if (malloc_outside_capture(reinterpret_cast<void**>(&w.partial), kSkSlotBytes * slots) !=
        cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (malloc_outside_capture(reinterpret_cast<void**>(&w.flags), 2 * sizeof(uint32_t) * slots) !=
            cudaSuccess ||
        cudaMemsetAsync(w.flags, 0, 2 * sizeof(uint32_t) * slots, stream) != cudaSuccess) {
        cudaGetLastError();
        g_retired.push_back(w.partial);  // not freed: cudaFree is as unsafe during a capture
        if (w.flags != nullptr) g_retired.push_back(w.flags);
        return nullptr;
    }
    w.slots = slots;
    if (it != g_sk.end()) {  // a grid with more pairs than the stream's earlier launches
        g_retired.push_back(it->second.partial);
        g_retired.push_back(it->second.flags);
    }
    return &(g_sk[key] = w);
}

// Device pair list of a contiguous problem whose row tiles outnumber the kernel's
// shared-memory list: one region of `stride` ints per CTA of a grid of at most `ctas`
// CTAs, kept per (device, stream) and grown on demand -- not while the stream is
// capturing a graph (cudaMalloc is not captured), where the caller falls back or fails.
struct ListWorkspace {
    int* buf = nullptr;
    int64_t ints = 0;
};
std::map<std::pair<int, void*>, ListWorkspace> g_list;

struct PairList {
    int* buf = nullptr;
    int stride = 0;
};

bool pair_list_workspace(int dev, cudaStream_t stream, int ctas, int64_t m_tiles, PairList* out) {
    const int64_t stride = (m_tiles + 1 + 31) / 32 * 32;
    const int64_t ints = stride * ctas;
    auto key = std::make_pair(dev, static_cast<void*>(stream));
    auto it = g_list.find(key);
    if (it == g_list.end() || it->second.ints < ints) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
            cudaGetLastError();
            return false;
        }
        const int64_t size = std::max(2 * ints, it == g_list.end() ? 0 : 2 * it->second.ints);
        ListWorkspace w;
        if (malloc_outside_capture(reinterpret_cast<void**>(&w.buf), sizeof(int) * size) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        w.ints = size;
        if (it != g_list.end()) {
            g_retired.push_back(it->second.buf);
            it->second = w;
        } else {
            it = g_list.emplace(key, w).first;
        }
    }
    out->buf = it->second.buf;
    out->stride = static_cast<int>(stride);
    return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Scale images of the E4M3 CTA-pair kernel (scale_pack.cuh), one buffer per
// (device, stream) like the stream-K scratch: launches on one stream run one after
// another (the pre-pass of the next call waits for the GEMM before it), launches on
// different streams may overlap and must not share it.  Grown on demand like the
// pair list, not while the stream is capturing a graph (cudaMalloc is not
// captured): then the GEMM converts the fp32 scales itself (same results).
struct PackWorkspace {
    uint32_t* buf = nullptr;
    int64_t words = 0;
};
std::map<std::pair<int, void*>, PackWorkspace> g_pack;

uint32_t* pack_workspace(int dev, cudaStream_t stream, int64_t words) {
    auto key = std::make_pair(dev, static_cast<void*>(stream));
    auto it = g_pack.find(key);
    if (it != g_pack.end() && it->second.words >= words) return it->second.buf;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return nullptr;
    }
    const int64_t size = std::max(2 * words, it == g_pack.end() ? 0 : 2 * it->second.words);
    PackWorkspace w;
    if (malloc_outside_capture(reinterpret_cast<void**>(&w.buf), sizeof(uint32_t) * size) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    w.words = size;
    if (it != g_pack.end()) g_retired.push_back(it->second.buf);
    return (g_pack[key] = w).buf;
}

// Resolve the current device and its cached state (lock held by caller).
int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        st.sms = sms;
        st.status = (major == 10 && minor == 3) ? FP8BS_OK : FP8BS_ERR_UNSUPPORTED;
        if (st.status == FP8BS_OK) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_fp8bs_error_word) != cudaSuccess) {
                cudaGetLastError();
                return FP8BS_ERR_CUDA;
            }
            st.err = static_cast<uint32_t*>(addr);
        }
        if (g_encode == nullptr) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr) {
                cudaGetLastError();
                return FP8BS_ERR_CUDA;
            }
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        st.ready = true;
    }
    *out = &st;
    return st.status;
}

// 2-D E4M3 tensor map: `outer` rows of `inner` bytes, box 128 bytes x box_outer
// rows, 128-byte swizzle, out-of-range rows read as zero.
int get_map(int dev, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer,
            const CUtensorMap** out) {
    MapKey key{dev, ptr, inner, outer, box_outer, 0};
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
        *out = &it->second;
        return FP8BS_OK;
    }
    CUtensorMap map;
    std::memset(&map, 0, sizeof(map));
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};  // bytes between rows
    cuuint32_t box[2] = {128u, box_outer};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return FP8BS_ERR_CUDA;
    if (g_maps.size() > 4096) g_maps.clear();
    auto ins = g_maps.emplace(key, map);
    *out = &ins.first->second;
    return FP8BS_OK;
}

// 3-D E4M3 tensor map over the same [outer rows, inner bytes] matrix viewed as
// [inner/128 K blocks][outer rows][128 bytes]: a box of 128 bytes x box_outer
// rows x box_kb K blocks lands in shared memory as box_kb consecutive
// 128-byte-swizzled [box_outer x 128 B] tiles.
int get_map3(int dev, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer,
             uint32_t box_kb, const CUtensorMap** out) {
    MapKey key{dev, ptr, inner, outer, box_outer, box_kb};
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
        *out = &it->second;
        return FP8BS_OK;
    }
    CUtensorMap map;
    std::memset(&map, 0, sizeof(map));
    cuuint64_t dims[3] = {128u, outer, inner / 128u};
    cuuint64_t strides[2] = {inner, 128u};  // bytes between rows, between K blocks
    cuuint32_t box[3] = {128u, box_outer, box_kb};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return FP8BS_ERR_CUDA;
    if (g_maps.size() > 4096) g_maps.clear();
    auto ins = g_maps.emplace(key, map);
    *out = &ins.first->second;
    return FP8BS_OK;
}

// Programmatic dependent launch: every kernel executes griddepcontrol.wait
// before it touches device memory, so it may be scheduled while the grid it
// follows in the stream is still finishing (its CTAs start on the SMs that
// grid has already freed); after a grid that never signals, or after a
// non-kernel stream operation, the launch is ordered as usual.
std::atomic<uint32_t> g_debug_flags{0};  // fp8bs_set_debug_flags (tests only)
// FP8BS_DEBUG_SINGLE_CTA: host-side routing of the plain entry points to the
// single-CTA kernel, so that tests can compare both kernels on one problem
constexpr uint32_t kDebugSingleCta = 0x2u;

inline void set_pdl(cudaLaunchAttribute& a) {
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
}

// Makes the scale images of an E4M3 pair-kernel call and points `p` at them; with
// no workspace to be had, leaves `p` without them (the kernel converts the fp32
// scales itself).  Only for row-major activation scales: there the kernel's own
// fetch is a gather of 4-byte values a row stride apart (one memory request per
// row and K block), which the images turn into three contiguous 512-byte copies a
// step; a transposed layout already gives contiguous 512-byte rows, and the extra
// launch (which must wait for the previous kernel) costs more than it saves.
// p.sa/sb/row_info, strides, rows, kb_count, nb_count, num_groups and num_m_tiles
// must be set.
int prepare_scale_images(DeviceState& st, int dev, GemmParams& p, bool masked, cudaStream_t stream) {
    if (p.sa_row_stride == 1) return FP8BS_OK;  // transposed, or one K block
    const int steps = (p.kb_count + fp8bs::PairLayout::kKbPerStage - 1) / fp8bs::PairLayout::kKbPerStage;
    const int64_t tiles = masked ? static_cast<int64_t>(p.num_groups) * p.num_m_tiles : p.num_m_tiles;
    const int64_t a_words = tiles * steps * 128;
    const int64_t b_words = static_cast<int64_t>(p.num_groups) * p.nb_count * steps * 128;
    if ((a_words + b_words) / 4 >= (int64_t{1} << 31)) return FP8BS_OK;  // 32-bit vector index
    uint32_t* buf = pack_workspace(dev, stream, a_words + b_words);
    if (buf == nullptr) return FP8BS_OK;
    fp8bs::ScalePackParams q{};
    q.sa = p.sa;
    q.sb = p.sb;
    q.row_info = p.row_info;
    q.packed_a = buf;
    q.packed_b = buf + a_words;
    q.err = p.err;
    q.rows = p.rows;
    q.sa_g_stride = p.sa_g_stride;
    q.sa_kb_stride = p.sa_kb_stride;
    q.sa_row_stride = p.sa_row_stride;
    q.a_vecs = static_cast<uint32_t>(a_words / 4);
    q.b_vecs = static_cast<uint32_t>(b_words / 4);
    q.kb_count = p.kb_count;
    q.steps = steps;
    q.tiles_per_group = p.num_m_tiles;
    q.masked = masked ? 1 : 0;
    const int64_t blocks = ((a_words + b_words) / 4 + 255) / 256;
    const int64_t max_blocks = static_cast<int64_t>(st.sms) * 8;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl(attr[0]);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks < max_blocks ? blocks : max_blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fp8bs::scale_pack_kernel, q) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    p.sf_a_packed = q.packed_a;
    p.sf_b_packed = q.packed_b;
    p.sf_steps = steps;
    return FP8BS_OK;
}

template <int BN, typename OutT, bool kMasked>
int launch(DeviceState& st, int attr_slot, const CUtensorMap& ta, const CUtensorMap& tb,
           const GemmParams& p, int64_t tiles_bound, cudaStream_t stream) {
    using L = SmemLayout<BN>;
    auto kern = fp8bs::grouped_gemm_kernel<BN, OutT, kMasked>;
    const int smem = (kMasked ? L::kBytesMasked : L::kBytesContiguous) + L::kAlignSlack;
    if (!st.attr_set[attr_slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        st.attr_set[attr_slot] = true;
    }
    const int grid = static_cast<int>(tiles_bound < st.sms ? tiles_bound : st.sms);
    if (grid <= 0) return FP8BS_OK;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl(attr[0]);
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(fp8bs::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, p) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return FP8BS_OK;
}

// CTA-pair kernel: cluster of 2, persistent over at most the number of pairs
// that fit on the device at once.
template <typename OutT, bool kMasked, bool kSwiglu = false, bool kMx = false>
int launch_pair(DeviceState& st, int attr_slot, const CUtensorMap& ta, const CUtensorMap& tb,
                const GemmParams& p, int64_t units_bound, cudaStream_t stream) {
    using L = fp8bs::PairLayoutT<kMx>;
    auto kern = fp8bs::grouped_gemm_pair_kernel<OutT, kMasked, kSwiglu, kMx>;
    const int smem = L::kBytes + L::kAlignSlack;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl(attr[1]);
    cfg.blockDim = dim3(fp8bs::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query sees the cluster shape only
    if (!st.attr_set[attr_slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        cfg.gridDim = dim3(2 * (st.sms / 2), 1, 1);
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) {
            cudaGetLastError();
            clusters = st.sms / 2;
        }
        st.max_clusters[attr_slot] = clusters;
        st.attr_set[attr_slot] = true;
    }
    const int64_t pairs = units_bound < st.max_clusters[attr_slot] ? units_bound
                                                                   : st.max_clusters[attr_slot];
    if (pairs <= 0) return FP8BS_OK;
    GemmParams q = p;
    q.debug_flags = g_debug_flags.load(std::memory_order_relaxed);
    int dev = 0;
    cudaGetDevice(&dev);
    SkWorkspace* w = kMasked ? nullptr : sk_workspace(dev, stream, 2 * st.max_clusters[attr_slot]);
    if (w != nullptr) {
        q.sk_partial = w->partial;
        q.sk_flags = w->flags;
        q.sk_slots = w->slots;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, q) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return FP8BS_OK;
}

// Software-promotion kernel (arbitrary fp32 scales): cluster of 2, 384 threads,
// round-robin units, no scratch.
template <typename OutT, bool kMasked>
int launch_promote(DeviceState& st, int attr_slot, const CUtensorMap& ta, const CUtensorMap& tb,
                   const GemmParams& p, int64_t units_bound, cudaStream_t stream) {
    using L = fp8bs::PromoteLayout;
    auto kern = fp8bs::grouped_gemm_promote_kernel<OutT, kMasked>;
    const int smem = L::kBytes + L::kAlignSlack;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl(attr[1]);
    cfg.blockDim = dim3(fp8bs::kPromoteThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query sees the cluster shape only
    if (!st.attr_set[attr_slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        cfg.gridDim = dim3(2 * (st.sms / 2), 1, 1);
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) {
            cudaGetLastError();
            clusters = st.sms / 2;
        }
        st.max_clusters[attr_slot] = clusters;
        st.attr_set[attr_slot] = true;
    }
    const int64_t pairs = units_bound < st.max_clusters[attr_slot] ? units_bound
                                                                   : st.max_clusters[attr_slot];
    if (pairs <= 0) return FP8BS_OK;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, p) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return FP8BS_OK;
}

template <bool kMasked>
int dispatch_pair(DeviceState& st, int out_dtype, const CUtensorMap& ta, const CUtensorMap& tb,
                  const GemmParams& p, int64_t units_bound, cudaStream_t stream) {
    // The masked (decode) variant streams each B tile once for all the m-tiles of its
    // group; splitting units across pairs would fetch it again later, so it stays
    // round-robin and needs no scratch.
    const int slot = 16 + (kMasked ? 2 : 0) + out_dtype;
    return out_dtype == FP8BS_OUT_BF16
               ? launch_pair<__nv_bfloat16, kMasked>(st, slot, ta, tb, p, units_bound, stream)
               : launch_pair<__half, kMasked>(st, slot, ta, tb, p, units_bound, stream);
}

template <bool kMasked>
int dispatch(DeviceState& st, int bn, int out_dtype, const CUtensorMap& ta, const CUtensorMap& tb,
             const GemmParams& p, int64_t tiles_bound, cudaStream_t stream) {
    const int slot = (kMasked ? 8 : 0) + (bn == 256 ? 4 : 0) + out_dtype;
    if (bn == 256) {
        return out_dtype == FP8BS_OUT_BF16
                   ? launch<256, __nv_bfloat16, kMasked>(st, slot, ta, tb, p, tiles_bound, stream)
                   : launch<256, __half, kMasked>(st, slot, ta, tb, p, tiles_bound, stream);
    }
    return out_dtype == FP8BS_OUT_BF16
               ? launch<128, __nv_bfloat16, kMasked>(st, slot, ta, tb, p, tiles_bound, stream)
               : launch<128, __half, kMasked>(st, slot, ta, tb, p, tiles_bound, stream);
}

// Checks shared by both variants; touches no CUDA state.
int validate_common(const void* a, const float* sa, int sa_layout, int64_t ld_sa, const void* b,
                    const float* sb, const void* d, int out_dtype, int64_t sa_rows, int64_t n,
                    int64_t k, int64_t num_groups) {
    if (n <= 0 || k <= 0 || n % 128 || k % 128) return FP8BS_ERR_INVALID_ARG;
    if (num_groups < 1) return FP8BS_ERR_INVALID_ARG;
    if (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F16) return FP8BS_ERR_INVALID_ARG;
    if (sa_layout != FP8BS_SA_MK && sa_layout != FP8BS_SA_KM) return FP8BS_ERR_INVALID_ARG;
    if (!a || !sa || !b || !sb || !d) return FP8BS_ERR_INVALID_ARG;
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(d, 16)) return FP8BS_ERR_INVALID_ARG;
    if (!aligned(sa, 4) || !aligned(sb, 4)) return FP8BS_ERR_INVALID_ARG;
    if (sa_layout == FP8BS_SA_KM) {
        if (ld_sa < sa_rows || ld_sa % 4 || !aligned(sa, 16)) return FP8BS_ERR_INVALID_ARG;
    }
    // TMA coordinates and tile indices are 32-bit
    if (num_groups * n > INT32_MAX || k > INT32_MAX / 2) return FP8BS_ERR_INVALID_ARG;
    return FP8BS_OK;
}

int pick_bn(int64_t n) { return n % 256 == 0 ? 256 : 128; }

}  // namespace

// ---------------------------------------------------------------------------
// Scratch of gemm_grouped_contiguous_noalloc: the stream-K partial tiles and
// slot counters of the CTA-pair kernel in one statically sized device array,
// for callers that may not allocate device memory.  Every GPU that loads this
// library holds it until the process exits.
namespace {
constexpr int kNoAllocSlots = 160;  // 2 per CTA pair, up to 80 pairs
constexpr size_t kNoAllocPartialBytes = kNoAllocSlots * kSkSlotBytes;
constexpr size_t kNoAllocFlagBytes = 2 * sizeof(uint32_t) * kNoAllocSlots;
}  // namespace
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocPartialBytes + kNoAllocFlagBytes];

namespace {

struct NoAllocDevice {
    bool ready = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
    bool attr_set[2] = {};
    int max_clusters[2] = {};
};
NoAllocDevice g_noalloc[kMaxDevices];

// 2-D/3-D maps are encoded on the stack for every call (no cache, no host heap).
int encode_map3_noalloc(const void* ptr, uint64_t inner, uint64_t outer, CUtensorMap* map) {
    std::memset(map, 0, sizeof(*map));
    cuuint64_t dims[3] = {128u, outer, inner / 128u};
    cuuint64_t strides[2] = {inner, 128u};
    cuuint32_t box[3] = {128u, 128u, static_cast<cuuint32_t>(fp8bs::PairLayout::kKbPerStage)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8BS_OK : FP8BS_ERR_CUDA;
}

template <typename OutT>
int launch_pair_noalloc(DeviceState& st, NoAllocDevice& nd, int slot, const CUtensorMap& ta,
                        const CUtensorMap& tb, GemmParams q, int64_t units_bound,
                        cudaStream_t stream) {
    using L = fp8bs::PairLayout;
    auto kern = fp8bs::grouped_gemm_pair_kernel<OutT, false, false>;
    const int smem = L::kBytes + L::kAlignSlack;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl(attr[1]);
    cfg.blockDim = dim3(fp8bs::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query sees the cluster shape only
    if (!nd.attr_set[slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        cfg.gridDim = dim3(2 * (st.sms / 2), 1, 1);
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) {
            cudaGetLastError();
            clusters = st.sms / 2;
        }
        nd.max_clusters[slot] = clusters;
        nd.attr_set[slot] = true;
    }
    // at most the pairs the array has stream-K slots for (2 each); a persistent grid of
    // fewer pairs is as correct, only less parallel
    int64_t pairs = units_bound < nd.max_clusters[slot] ? units_bound : nd.max_clusters[slot];
    if (pairs > kNoAllocSlots / 2) pairs = kNoAllocSlots / 2;
    if (pairs <= 0) return FP8BS_OK;
    // the slot counters must start at zero; a launch that gave up could have left
    // them set, so clear them on the stream before every launch (a non-kernel stream
    // operation: the launch then cannot overlap the tail of the preceding kernel)
    uint32_t* flags = reinterpret_cast<uint32_t*>(nd.scratch + kNoAllocPartialBytes);
    if (cudaMemsetAsync(flags, 0, kNoAllocFlagBytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    q.debug_flags = g_debug_flags.load(std::memory_order_relaxed);
    q.sk_partial = reinterpret_cast<float*>(nd.scratch);
    q.sk_flags = flags;
    q.sk_slots = kNoAllocSlots;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, q) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return FP8BS_OK;
}

}  // namespace

extern "C" {

int fp8bs_abi_version(void) { return 1; }

uint64_t fp8bs_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int fp8bs_set_debug_flags(uint32_t flags) {
    if (flags & ~(fp8bs::kDebugStallMma | kDebugSingleCta)) return FP8BS_ERR_INVALID_ARG;
    g_debug_flags.store(flags, std::memory_order_relaxed);
    return FP8BS_OK;
}

const char* fp8bs_status_string(int status) {
    switch (status) {
        case FP8BS_OK: return "ok";
        case FP8BS_ERR_INVALID_ARG: return "invalid argument";
        case FP8BS_ERR_UNSUPPORTED: return "unsupported device (needs compute capability 10.3)";
        case FP8BS_ERR_CUDA: return "CUDA error";
        case FP8BS_ERR_DEVICE: return "device error word set";
        default: return "unknown status";
    }
}

int fp8bs_clear_cache(void) {
    std::lock_guard<std::mutex> lock(g_mutex);
    g_maps.clear();
    return FP8BS_OK;
}

int gemm_grouped_contiguous(const void* a, const float* scale_a, int sa_layout, int64_t ld_sa,
                            const void* b, const float* scale_b, const int32_t* grouped_layout,
                            void* d, int out_dtype, int64_t m_sum, int64_t n, int64_t k,
                            int64_t num_groups, void* stream) {
    if (m_sum < 0 || m_sum > INT32_MAX - 128) return FP8BS_ERR_INVALID_ARG;
    if (m_sum == 0) {
        // nothing to compute; still reject malformed sizes and codes
        if (n <= 0 || k <= 0 || n % 128 || k % 128 || num_groups < 1 ||
            (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F16) ||
            (sa_layout != FP8BS_SA_MK && sa_layout != FP8BS_SA_KM))
            return FP8BS_ERR_INVALID_ARG;
        return FP8BS_OK;
    }
    int v = validate_common(a, scale_a, sa_layout, ld_sa, b, scale_b, d, out_dtype, m_sum, n, k,
                            num_groups);
    if (v != FP8BS_OK) return v;
    if (!grouped_layout || !aligned(grouped_layout, 4)) return FP8BS_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != FP8BS_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t m_tiles = (m_sum + 127) / 128;
    bool pair = m_tiles <= fp8bs::kPairMaxTilesWs &&
                num_groups < fp8bs::kPairMaxGroups &&
                !(g_debug_flags.load(std::memory_order_relaxed) & kDebugSingleCta);
    // a pair list longer than shared memory holds goes to a device workspace; without
    // one (a first such call while capturing a graph) the single-CTA kernel runs
    PairList plist;
    if (pair && m_tiles > fp8bs::kPairMaxTiles &&
        !pair_list_workspace(dev, static_cast<cudaStream_t>(stream), st->sms, m_tiles, &plist))
        pair = false;
    const int bn = pair ? 256 : pick_bn(n);
    const CUtensorMap *ta = nullptr, *tb = nullptr;
    constexpr uint32_t kKbBox = fp8bs::PairLayout::kKbPerStage;
    if (pair) {
        if ((rc = get_map3(dev, a, k, m_sum, 128, kKbBox, &ta)) != FP8BS_OK) return rc;
        if ((rc = get_map3(dev, b, k, num_groups * n, 128, kKbBox, &tb)) != FP8BS_OK) return rc;
    } else {
        if ((rc = get_map(dev, a, k, m_sum, 128, &ta)) != FP8BS_OK) return rc;
        if ((rc = get_map(dev, b, k, num_groups * n, bn, &tb)) != FP8BS_OK) return rc;
    }

    GemmParams p{};
    p.sa = scale_a;
    p.sb = scale_b;
    p.row_info = grouped_layout;
    p.d = d;
    p.err = st->err;
    p.rows = m_sum;
    p.sa_g_stride = 0;
    p.sa_kb_stride = sa_layout == FP8BS_SA_KM ? ld_sa : 1;
    p.sa_row_stride = sa_layout == FP8BS_SA_KM ? 1 : k / 128;
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_groups = static_cast<int>(num_groups);
    p.kb_count = static_cast<int>(k / 128);
    p.nb_count = static_cast<int>(n / 128);
    p.num_m_tiles = static_cast<int>((m_sum + 127) / 128);
    // the pair kernel runs n % 256 == 128 with a 128-column last tile
    p.num_n_tiles = static_cast<int>(pair ? (n + 255) / 256 : n / bn);
    p.n_half = pair && n % 256 != 0 ? 1 : 0;
    p.raster_band = 8;
    p.list_ws = plist.buf;
    p.list_ws_stride = plist.stride;
    p.d_align16 = aligned(d, 32) ? 0 : 1;
    const int64_t tiles = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
    if (pair) {
        if ((rc = prepare_scale_images(*st, dev, p, false, static_cast<cudaStream_t>(stream))) != FP8BS_OK)
            return rc;
        return dispatch_pair<false>(*st, out_dtype, *ta, *tb, p, tiles,
                                    static_cast<cudaStream_t>(stream));
    }
    return dispatch<false>(*st, bn, out_dtype, *ta, *tb, p, tiles,
                           static_cast<cudaStream_t>(stream));
}

int gemm_grouped_masked(const void* a, const float* scale_a, int sa_layout, int64_t ld_sa,
                        const void* b, const float* scale_b, const int32_t* masked_m,
                        int64_t expected_m, void* d, int out_dtype, int64_t num_groups,
                        int64_t m_max, int64_t n, int64_t k, void* stream) {
    (void)expected_m;  // scheduling hint only; results never depend on it
    if (m_max < 0 || num_groups < 1 || num_groups > fp8bs::kMaxMaskedGroups)
        return FP8BS_ERR_INVALID_ARG;
    if (m_max > 0 && num_groups * m_max > INT32_MAX - 128) return FP8BS_ERR_INVALID_ARG;
    if (m_max == 0) {
        if (n <= 0 || k <= 0 || n % 128 || k % 128 ||
            (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F16) ||
            (sa_layout != FP8BS_SA_MK && sa_layout != FP8BS_SA_KM))
            return FP8BS_ERR_INVALID_ARG;
        return FP8BS_OK;
    }
    int v = validate_common(a, scale_a, sa_layout, ld_sa, b, scale_b, d, out_dtype, m_max, n, k,
                            num_groups);
    if (v != FP8BS_OK) return v;
    if (!masked_m || !aligned(masked_m, 4)) return FP8BS_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != FP8BS_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const bool pair = !(g_debug_flags.load(std::memory_order_relaxed) & kDebugSingleCta);
    const int bn = pair ? 256 : pick_bn(n);
    const CUtensorMap *ta = nullptr, *tb = nullptr;
    constexpr uint32_t kKbBox = fp8bs::PairLayout::kKbPerStage;
    if (pair) {
        if ((rc = get_map3(dev, a, k, num_groups * m_max, 128, kKbBox, &ta)) != FP8BS_OK) return rc;
        if ((rc = get_map3(dev, b, k, num_groups * n, 128, kKbBox, &tb)) != FP8BS_OK) return rc;
    } else {
        if ((rc = get_map(dev, a, k, num_groups * m_max, 128, &ta)) != FP8BS_OK) return rc;
        if ((rc = get_map(dev, b, k, num_groups * n, bn, &tb)) != FP8BS_OK) return rc;
    }

    const int64_t kb = k / 128;
    GemmParams p{};
    p.sa = scale_a;
    p.sb = scale_b;
    p.row_info = masked_m;
    p.d = d;
    p.err = st->err;
    p.rows = m_max;
    p.sa_g_stride = sa_layout == FP8BS_SA_KM ? kb * ld_sa : m_max * kb;
    p.sa_kb_stride = sa_layout == FP8BS_SA_KM ? ld_sa : 1;
    p.sa_row_stride = sa_layout == FP8BS_SA_KM ? 1 : kb;
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_groups = static_cast<int>(num_groups);
    p.kb_count = static_cast<int>(kb);
    p.nb_count = static_cast<int>(n / 128);
    p.num_m_tiles = static_cast<int>((m_max + 127) / 128);
    p.num_n_tiles = static_cast<int>(pair ? (n + 255) / 256 : n / bn);
    p.n_half = pair && n % 256 != 0 ? 1 : 0;
    p.raster_band = 1;
    p.d_align16 = aligned(d, 32) ? 0 : 1;
    if (pair) {
        const int64_t units = num_groups * ((m_max + 255) / 256) * p.num_n_tiles;
        if ((rc = prepare_scale_images(*st, dev, p, true, static_cast<cudaStream_t>(stream))) != FP8BS_OK)
            return rc;
        return dispatch_pair<true>(*st, out_dtype, *ta, *tb, p, units,
                                   static_cast<cudaStream_t>(stream));
    }
    const int64_t tiles = num_groups * p.num_m_tiles * p.num_n_tiles;
    return dispatch<true>(*st, bn, out_dtype, *ta, *tb, p, tiles,
                          static_cast<cudaStream_t>(stream));
}

// Output scales of the fused gate/up epilogue: [rows, n/256] (MK) or the
// transposed [n/256, ld] (KM), the two activation-scale layouts the grouped
// GEMM itself accepts, so the result feeds the down projection directly.
static int validate_out_scale(const float* out_scale, int layout, int64_t ld, int64_t rows) {
    if (!out_scale || !aligned(out_scale, 4)) return FP8BS_ERR_INVALID_ARG;
    if (layout == FP8BS_SA_MK) return FP8BS_OK;
    if (layout != FP8BS_SA_KM) return FP8BS_ERR_INVALID_ARG;
    if (ld < rows || ld % 4 || !aligned(out_scale, 16)) return FP8BS_ERR_INVALID_ARG;
    return FP8BS_OK;
}

int gemm_grouped_contiguous_silu_mul_quant(const void* a, const float* scale_a, int sa_layout,
                                           int64_t ld_sa, const void* b, const float* scale_b,
                                           const int32_t* grouped_layout, void* out,
                                           float* out_scale, int out_scale_layout,
                                           int64_t ld_out_scale, int64_t m_sum, int64_t n,
                                           int64_t k, int64_t num_groups, void* stream) {
    if (m_sum < 0 || m_sum > INT32_MAX - 128) return FP8BS_ERR_INVALID_ARG;
    if (n <= 0 || k <= 0 || n % 256 || k % 128 || num_groups < 1) return FP8BS_ERR_INVALID_ARG;
    if ((sa_layout != FP8BS_SA_MK && sa_layout != FP8BS_SA_KM) ||
        (out_scale_layout != FP8BS_SA_MK && out_scale_layout != FP8BS_SA_KM))
        return FP8BS_ERR_INVALID_ARG;
    if (m_sum == 0) return FP8BS_OK;
    int v = validate_common(a, scale_a, sa_layout, ld_sa, b, scale_b, out, FP8BS_OUT_BF16, m_sum,
                            n, k, num_groups);
    if (v != FP8BS_OK) return v;
    if ((v = validate_out_scale(out_scale, out_scale_layout, ld_out_scale, m_sum)) != FP8BS_OK)
        return v;
    if (!grouped_layout || !aligned(grouped_layout, 4) || !aligned(out, 32))
        return FP8BS_ERR_INVALID_ARG;
    const int64_t m_tiles = (m_sum + 127) / 128;
    if (m_tiles > fp8bs::kPairMaxTilesWs || num_groups >= fp8bs::kPairMaxGroups)
        return FP8BS_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != FP8BS_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    PairList plist;
    if (m_tiles > fp8bs::kPairMaxTiles &&
        !pair_list_workspace(dev, static_cast<cudaStream_t>(stream), st->sms, m_tiles, &plist))
        return FP8BS_ERR_CUDA;  // a first call this large while the stream captures a graph
    const CUtensorMap *ta = nullptr, *tb = nullptr;
    constexpr uint32_t kKbBox = fp8bs::PairLayout::kKbPerStage;
    if ((rc = get_map3(dev, a, k, m_sum, 128, kKbBox, &ta)) != FP8BS_OK) return rc;
    if ((rc = get_map3(dev, b, k, num_groups * n, 128, kKbBox, &tb)) != FP8BS_OK) return rc;

    GemmParams p{};
    p.sa = scale_a;
    p.sb = scale_b;
    p.row_info = grouped_layout;
    p.d = out;
    p.err = st->err;
    p.rows = m_sum;
    p.sa_g_stride = 0;
    p.sa_kb_stride = sa_layout == FP8BS_SA_KM ? ld_sa : 1;
    p.sa_row_stride = sa_layout == FP8BS_SA_KM ? 1 : k / 128;
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_groups = static_cast<int>(num_groups);
    p.kb_count = static_cast<int>(k / 128);
    p.nb_count = static_cast<int>(n / 128);
    p.num_m_tiles = static_cast<int>(m_tiles);
    p.num_n_tiles = static_cast<int>(n / 256);  // 128-column output blocks
    p.raster_band = 8;
    p.q_scale = out_scale;
    p.qs_g_stride = 0;
    p.qs_row_stride = out_scale_layout == FP8BS_SA_KM ? 1 : n / 256;
    p.qs_col_stride = out_scale_layout == FP8BS_SA_KM ? ld_out_scale : 1;
    p.list_ws = plist.buf;
    p.list_ws_stride = plist.stride;
    if ((rc = prepare_scale_images(*st, dev, p, false, static_cast<cudaStream_t>(stream))) != FP8BS_OK)
        return rc;
    return launch_pair<__nv_bfloat16, false, true>(*st, 24, *ta, *tb, p,
                                                   m_tiles * p.num_n_tiles,
                                                   static_cast<cudaStream_t>(stream));
}

int gemm_grouped_masked_silu_mul_quant(const void* a, const float* scale_a, int sa_layout,
                                       int64_t ld_sa, const void* b, const float* scale_b,
                                       const int32_t* masked_m, int64_t expected_m, void* out,
                                       float* out_scale, int out_scale_layout,
                                       int64_t ld_out_scale, int64_t num_groups, int64_t m_max,
                                       int64_t n, int64_t k, void* stream) {
    (void)expected_m;  // scheduling hint only; results never depend on it
    if (m_max < 0 || num_groups < 1 || num_groups > fp8bs::kMaxMaskedGroups)
        return FP8BS_ERR_INVALID_ARG;
    if (m_max > 0 && num_groups * m_max > INT32_MAX - 128) return FP8BS_ERR_INVALID_ARG;
    if (n <= 0 || k <= 0 || n % 256 || k % 128) return FP8BS_ERR_INVALID_ARG;
    if ((sa_layout != FP8BS_SA_MK && sa_layout != FP8BS_SA_KM) ||
        (out_scale_layout != FP8BS_SA_MK && out_scale_layout != FP8BS_SA_KM))
        return FP8BS_ERR_INVALID_ARG;
    if (m_max == 0) return FP8BS_OK;
    int v = validate_common(a, scale_a, sa_layout, ld_sa, b, scale_b, out, FP8BS_OUT_BF16, m_max,
                            n, k, num_groups);
    if (v != FP8BS_OK) return v;
    if ((v = validate_out_scale(out_scale, out_scale_layout, ld_out_scale, m_max)) != FP8BS_OK)
        return v;
    if (!masked_m || !aligned(masked_m, 4) || !aligned(out, 32)) return FP8BS_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != FP8BS_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const CUtensorMap *ta = nullptr, *tb = nullptr;
    constexpr uint32_t kKbBox = fp8bs::PairLayout::kKbPerStage;
    if ((rc = get_map3(dev, a, k, num_groups * m_max, 128, kKbBox, &ta)) != FP8BS_OK) return rc;
    if ((rc = get_map3(dev, b, k, num_groups * n, 128, kKbBox, &tb)) != FP8BS_OK) return rc;

    const int64_t kb = k / 128;
    const int64_t blocks = n / 256;
    GemmParams p{};
    p.sa = scale_a;
    p.sb = scale_b;
    p.row_info = masked_m;
    p.d = out;
    p.err = st->err;
    p.rows = m_max;
    p.sa_g_stride = sa_layout == FP8BS_SA_KM ? kb * ld_sa : m_max * kb;
    p.sa_kb_stride = sa_layout == FP8BS_SA_KM ? ld_sa : 1;
    p.sa_row_stride = sa_layout == FP8BS_SA_KM ? 1 : kb;
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_groups = static_cast<int>(num_groups);
    p.kb_count = static_cast<int>(kb);
    p.nb_count = static_cast<int>(n / 128);
    p.num_m_tiles = static_cast<int>((m_max + 127) / 128);
    p.num_n_tiles = static_cast<int>(blocks);
    p.raster_band = 1;
    p.q_scale = out_scale;
    p.qs_g_stride = out_scale_layout == FP8BS_SA_KM ? blocks * ld_out_scale : m_max * blocks;
    p.qs_row_stride = out_scale_layout == FP8BS_SA_KM ? 1 : blocks;
    p.qs_col_stride = out_scale_layout == FP8BS_SA_KM ? ld_out_scale : 1;
    const int64_t units = num_groups * ((m_max + 255) / 256) * blocks;
    if ((rc = prepare_scale_images(*st, dev, p, true, static_cast<cudaStream_t>(stream))) != FP8BS_OK)
        return rc;
    return launch_pair<__nv_bfloat16, true, true>(*st, 25, *ta, *tb, p, units,
                                                  static_cast<cudaStream_t>(stream));
}

int gemm_grouped_contiguous_fp32_scales(const void* a, const float* scale_a, int sa_layout,
                                        int64_t ld_sa, const void* b, const float* scale_b,
                                        const int32_t* grouped_layout, void* d, int out_dtype,
                                        int64_t m_sum, int64_t n, int64_t k, int64_t num_groups,
                                        void* stream) {
    if (m_sum < 0 || m_sum > INT32_MAX - 128) return FP8BS_ERR_INVALID_ARG;
    if (n <= 0 || k <= 0 || n % 256 || k % 128 || num_groups < 1 ||
        (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F16) ||
        (sa_layout != FP8BS_SA_MK && sa_layout != FP8BS_SA_KM))
        return FP8BS_ERR_INVALID_ARG;
    if (m_sum == 0) return FP8BS_OK;
    int v = validate_common(a, scale_a, sa_layout, ld_sa, b, scale_b, d, out_dtype, m_sum, n, k,
                            num_groups);
    if (v != FP8BS_OK) return v;
    const int64_t m_tiles = (m_sum + 127) / 128;
    if (!grouped_layout || !aligned(grouped_layout, 4) || !aligned(d, 32) ||
        m_tiles > fp8bs::kPairMaxTilesWs || num_groups >= fp8bs::kPairMaxGroups)
        return FP8BS_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != FP8BS_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    PairList plist;
    if (m_tiles > fp8bs::kPairMaxTiles &&
        !pair_list_workspace(dev, static_cast<cudaStream_t>(stream), st->sms, m_tiles, &plist))
        return FP8BS_ERR_CUDA;  // a first call this large while the stream captures a graph
    const CUtensorMap *ta = nullptr, *tb = nullptr;
    constexpr uint32_t kKbBox = fp8bs::PromoteLayout::kKbPerStage;
    if ((rc = get_map3(dev, a, k, m_sum, 128, kKbBox, &ta)) != FP8BS_OK) return rc;
    if ((rc = get_map3(dev, b, k, num_groups * n, 128, kKbBox, &tb)) != FP8BS_OK) return rc;

    GemmParams p{};
    p.sa = scale_a;
    p.sb = scale_b;
    p.row_info = grouped_layout;
    p.d = d;
    p.err = st->err;
    p.rows = m_sum;
    p.sa_g_stride = 0;
    p.sa_kb_stride = sa_layout == FP8BS_SA_KM ? ld_sa : 1;
    p.sa_row_stride = sa_layout == FP8BS_SA_KM ? 1 : k / 128;
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_groups = static_cast<int>(num_groups);
    p.kb_count = static_cast<int>(k / 128);
    p.nb_count = static_cast<int>(n / 128);
    p.num_m_tiles = static_cast<int>(m_tiles);
    p.num_n_tiles = static_cast<int>(n / 256);
    p.raster_band = 8;
    p.list_ws = plist.buf;
    p.list_ws_stride = plist.stride;
    const int64_t units = m_tiles * p.num_n_tiles;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return out_dtype == FP8BS_OUT_BF16
               ? launch_promote<__nv_bfloat16, false>(*st, 26, *ta, *tb, p, units, s)
               : launch_promote<__half, false>(*st, 27, *ta, *tb, p, units, s);
}

int gemm_grouped_masked_fp32_scales(const void* a, const float* scale_a, int sa_layout,
                                    int64_t ld_sa, const void* b, const float* scale_b,
                                    const int32_t* masked_m, int64_t expected_m, void* d,
                                    int out_dtype, int64_t num_groups, int64_t m_max, int64_t n,
                                    int64_t k, void* stream) {
    (void)expected_m;  // scheduling hint only; results never depend on it
    if (m_max < 0 || num_groups < 1 || num_groups > fp8bs::kMaxMaskedGroups)
        return FP8BS_ERR_INVALID_ARG;
    if (m_max > 0 && num_groups * m_max > INT32_MAX - 128) return FP8BS_ERR_INVALID_ARG;
    if (n <= 0 || k <= 0 || n % 256 || k % 128 ||
        (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F16) ||
        (sa_layout != FP8BS_SA_MK && sa_layout != FP8BS_SA_KM))
        return FP8BS_ERR_INVALID_ARG;
    if (m_max == 0) return FP8BS_OK;
    int v = validate_common(a, scale_a, sa_layout, ld_sa, b, scale_b, d, out_dtype, m_max, n, k,
                            num_groups);
    if (v != FP8BS_OK) return v;
    if (!masked_m || !aligned(masked_m, 4) || !aligned(d, 32)) return FP8BS_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != FP8BS_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const CUtensorMap *ta = nullptr, *tb = nullptr;
    constexpr uint32_t kKbBox = fp8bs::PromoteLayout::kKbPerStage;
    if ((rc = get_map3(dev, a, k, num_groups * m_max, 128, kKbBox, &ta)) != FP8BS_OK) return rc;
    if ((rc = get_map3(dev, b, k, num_groups * n, 128, kKbBox, &tb)) != FP8BS_OK) return rc;

    const int64_t kb = k / 128;
    GemmParams p{};
    p.sa = scale_a;
    p.sb = scale_b;
    p.row_info = masked_m;
    p.d = d;
    p.err = st->err;
    p.rows = m_max;
    p.sa_g_stride = sa_layout == FP8BS_SA_KM ? kb * ld_sa : m_max * kb;
    p.sa_kb_stride = sa_layout == FP8BS_SA_KM ? ld_sa : 1;
    p.sa_row_stride = sa_layout == FP8BS_SA_KM ? 1 : kb;
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_groups = static_cast<int>(num_groups);
    p.kb_count = static_cast<int>(kb);
    p.nb_count = static_cast<int>(n / 128);
    p.num_m_tiles = static_cast<int>((m_max + 127) / 128);
    p.num_n_tiles = static_cast<int>(n / 256);
    p.raster_band = 1;
    const int64_t units = num_groups * ((m_max + 255) / 256) * p.num_n_tiles;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return out_dtype == FP8BS_OUT_BF16
               ? launch_promote<__nv_bfloat16, true>(*st, 28, *ta, *tb, p, units, s)
               : launch_promote<__half, true>(*st, 29, *ta, *tb, p, units, s);
}

// MXFP4 arguments shared by both variants: packed E2M1 operands (16-byte
// aligned for TMA), E8M0 scale bytes (4-byte aligned: copied a word at a time),
// 32-byte aligned output, n % 256 == 0, k % 256 == 0 (128 bytes per K block).
static int validate_mx(const void* a, const uint8_t* sa, const void* b, const uint8_t* sb,
                       const void* d, int out_dtype, int64_t n, int64_t k, int64_t num_groups) {
    if (n <= 0 || k <= 0 || n % 256 || k % 256 || num_groups < 1) return FP8BS_ERR_INVALID_ARG;
    if (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F16) return FP8BS_ERR_INVALID_ARG;
    if (!a || !sa || !b || !sb || !d) return FP8BS_ERR_INVALID_ARG;
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(d, 32) || !aligned(sa, 4) || !aligned(sb, 4))
        return FP8BS_ERR_INVALID_ARG;
    if (num_groups * n > INT32_MAX || k > INT32_MAX / 2) return FP8BS_ERR_INVALID_ARG;
    return FP8BS_OK;
}

int gemm_grouped_contiguous_mxfp4(const void* a, const uint8_t* scale_a, const void* b,
                                  const uint8_t* scale_b, const int32_t* grouped_layout, void* d,
                                  int out_dtype, int64_t m_sum, int64_t n, int64_t k,
                                  int64_t num_groups, void* stream) {
    if (m_sum < 0 || m_sum > INT32_MAX - 128) return FP8BS_ERR_INVALID_ARG;
    if (m_sum == 0) {
        if (n <= 0 || k <= 0 || n % 256 || k % 256 || num_groups < 1 ||
            (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F16))
            return FP8BS_ERR_INVALID_ARG;
        return FP8BS_OK;
    }
    int v = validate_mx(a, scale_a, b, scale_b, d, out_dtype, n, k, num_groups);
    if (v != FP8BS_OK) return v;
    const int64_t m_tiles = (m_sum + 127) / 128;
    if (!grouped_layout || !aligned(grouped_layout, 4) || m_tiles > fp8bs::kPairMaxTilesWs ||
        num_groups >= fp8bs::kPairMaxGroups)
        return FP8BS_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != FP8BS_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    PairList plist;
    if (m_tiles > fp8bs::kMxMaxTiles &&
        !pair_list_workspace(dev, static_cast<cudaStream_t>(stream), st->sms, m_tiles, &plist))
        return FP8BS_ERR_CUDA;  // a first call this large while the stream captures a graph
    const CUtensorMap *ta = nullptr, *tb = nullptr;
    constexpr uint32_t kKbBox = fp8bs::PairLayout::kKbPerStage;
    // packed rows: k/2 bytes, K blocks of 128 bytes
    if ((rc = get_map3(dev, a, k / 2, m_sum, 128, kKbBox, &ta)) != FP8BS_OK) return rc;
    if ((rc = get_map3(dev, b, k / 2, num_groups * n, 128, kKbBox, &tb)) != FP8BS_OK) return rc;

    GemmParams p{};
    p.sa = reinterpret_cast<const float*>(scale_a);  // E8M0 bytes; the MX kernel reads bytes
    p.sb = reinterpret_cast<const float*>(scale_b);
    p.row_info = grouped_layout;
    p.d = d;
    p.err = st->err;
    p.rows = m_sum;
    p.sa_g_stride = 0;
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_groups = static_cast<int>(num_groups);
    p.kb_count = static_cast<int>(k / 256);
    p.nb_count = static_cast<int>(n / 128);
    p.num_m_tiles = static_cast<int>(m_tiles);
    p.num_n_tiles = static_cast<int>(n / 256);
    p.raster_band = 8;
    p.list_ws = plist.buf;
    p.list_ws_stride = plist.stride;
    const int64_t tiles = m_tiles * p.num_n_tiles;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return out_dtype == FP8BS_OUT_BF16
               ? launch_pair<__nv_bfloat16, false, false, true>(*st, 20, *ta, *tb, p, tiles, s)
               : launch_pair<__half, false, false, true>(*st, 21, *ta, *tb, p, tiles, s);
}

int gemm_grouped_masked_mxfp4(const void* a, const uint8_t* scale_a, const void* b,
                              const uint8_t* scale_b, const int32_t* masked_m, int64_t expected_m,
                              void* d, int out_dtype, int64_t num_groups, int64_t m_max,
                              int64_t n, int64_t k, void* stream) {
    (void)expected_m;  // scheduling hint only; results never depend on it
    if (m_max < 0 || num_groups < 1 || num_groups > fp8bs::kMaxMaskedGroups)
        return FP8BS_ERR_INVALID_ARG;
    if (m_max > 0 && num_groups * m_max > INT32_MAX - 128) return FP8BS_ERR_INVALID_ARG;
    if (m_max == 0) {
        if (n <= 0 || k <= 0 || n % 256 || k % 256 ||
            (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F16))
            return FP8BS_ERR_INVALID_ARG;
        return FP8BS_OK;
    }
    int v = validate_mx(a, scale_a, b, scale_b, d, out_dtype, n, k, num_groups);
    if (v != FP8BS_OK) return v;
    if (!masked_m || !aligned(masked_m, 4)) return FP8BS_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != FP8BS_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const CUtensorMap *ta = nullptr, *tb = nullptr;
    constexpr uint32_t kKbBox = fp8bs::PairLayout::kKbPerStage;
    if ((rc = get_map3(dev, a, k / 2, num_groups * m_max, 128, kKbBox, &ta)) != FP8BS_OK) return rc;
    if ((rc = get_map3(dev, b, k / 2, num_groups * n, 128, kKbBox, &tb)) != FP8BS_OK) return rc;

    GemmParams p{};
    p.sa = reinterpret_cast<const float*>(scale_a);
    p.sb = reinterpret_cast<const float*>(scale_b);
    p.row_info = masked_m;
    p.d = d;
    p.err = st->err;
    p.rows = m_max;
    p.sa_g_stride = m_max * (k / 32);  // bytes between groups of scale_a
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_groups = static_cast<int>(num_groups);
    p.kb_count = static_cast<int>(k / 256);
    p.nb_count = static_cast<int>(n / 128);
    p.num_m_tiles = static_cast<int>((m_max + 127) / 128);
    p.num_n_tiles = static_cast<int>(n / 256);
    p.raster_band = 1;
    const int64_t units = num_groups * ((m_max + 255) / 256) * p.num_n_tiles;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return out_dtype == FP8BS_OUT_BF16
               ? launch_pair<__nv_bfloat16, true, false, true>(*st, 22, *ta, *tb, p, units, s)
               : launch_pair<__half, true, false, true>(*st, 23, *ta, *tb, p, units, s);
}

// Contiguous grouped GEMM that allocates nothing: the CTA-pair kernel with its
// stream-K scratch in g_noalloc_scratch instead of a cudaMalloc'd workspace.
int gemm_grouped_contiguous_noalloc(const void* a, const float* scale_a, int sa_layout,
                                    int64_t ld_sa, const void* b, const float* scale_b,
                                    const int32_t* grouped_layout, void* d, int out_dtype,
                                    int64_t m_sum, int64_t n, int64_t k, int64_t num_groups,
                                    void* stream) {
    if (m_sum < 0 || m_sum > INT32_MAX - 128) return FP8BS_ERR_INVALID_ARG;
    if (m_sum == 0) {
        if (n <= 0 || k <= 0 || n % 128 || k % 128 || num_groups < 1 ||
            (out_dtype != FP8BS_OUT_BF16 && out_dtype != FP8BS_OUT_F16) ||
            (sa_layout != FP8BS_SA_MK && sa_layout != FP8BS_SA_KM))
            return FP8BS_ERR_INVALID_ARG;
        return FP8BS_OK;
    }
    int v = validate_common(a, scale_a, sa_layout, ld_sa, b, scale_b, d, out_dtype, m_sum, n, k,
                            num_groups);
    if (v != FP8BS_OK) return v;
    if (!grouped_layout || !aligned(grouped_layout, 4)) return FP8BS_ERR_INVALID_ARG;
    // only shapes the CTA-pair kernel takes
    const int64_t m_tiles = (m_sum + 127) / 128;
    if (m_tiles > fp8bs::kPairMaxTiles || num_groups >= fp8bs::kPairMaxGroups)
        return FP8BS_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != FP8BS_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    NoAllocDevice& nd = g_noalloc[dev];
    if (!nd.ready) {
        // once per device, with that device current: the device address of the array
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        nd.scratch = static_cast<unsigned char*>(addr);
        nd.ready = true;
    }
    CUtensorMap ta, tb;
    if ((rc = encode_map3_noalloc(a, k, m_sum, &ta)) != FP8BS_OK) return rc;
    if ((rc = encode_map3_noalloc(b, k, num_groups * n, &tb)) != FP8BS_OK) return rc;

    GemmParams p{};
    p.sa = scale_a;
    p.sb = scale_b;
    p.row_info = grouped_layout;
    p.d = d;
    p.err = st->err;
    p.rows = m_sum;
    p.sa_g_stride = 0;
    p.sa_kb_stride = sa_layout == FP8BS_SA_KM ? ld_sa : 1;
    p.sa_row_stride = sa_layout == FP8BS_SA_KM ? 1 : k / 128;
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_groups = static_cast<int>(num_groups);
    p.kb_count = static_cast<int>(k / 128);
    p.nb_count = static_cast<int>(n / 128);
    p.num_m_tiles = static_cast<int>(m_tiles);
    p.num_n_tiles = static_cast<int>((n + 255) / 256);
    p.n_half = n % 256 != 0 ? 1 : 0;
    p.raster_band = 8;
    p.d_align16 = aligned(d, 32) ? 0 : 1;
    const int64_t tiles = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return out_dtype == FP8BS_OUT_BF16
               ? launch_pair_noalloc<__nv_bfloat16>(*st, nd, 0, ta, tb, p, tiles, s)
               : launch_pair_noalloc<__half>(*st, nd, 1, ta, tb, p, tiles, s);
}

int fp8bs_device_error(int device, uint32_t* flags) {
    if (!flags || device < 0 || device >= kMaxDevices) return FP8BS_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mutex);
    int old = 0;
    if (cudaGetDevice(&old) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    int rc = FP8BS_OK;
    uint32_t value = 0;
    const uint32_t zero = 0;
    if (cudaSetDevice(device) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&value, g_fp8bs_error_word, sizeof(value)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_fp8bs_error_word, &zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        rc = FP8BS_ERR_CUDA;
    }
    if (rc == FP8BS_OK && value != 0) {
        // a launch that gave up may have left stream-K slot counters half set
        for (auto& kv : g_sk)
            if (kv.first.first == device) cudaMemset(kv.second.flags, 0, 2 * sizeof(uint32_t) * kv.second.slots);
        cudaDeviceSynchronize();
        cudaGetLastError();
    }
    cudaSetDevice(old);
    *flags = value;
    if (rc == FP8BS_OK && value != 0) rc = FP8BS_ERR_DEVICE;
    return rc;
}

}  // extern "C"
