// C-ABI of libnvfp4gg: argument checks, tensor-map set-up and kernel launch
// for the masked, block-scaled NVFP4 grouped GEMM-NT (include/nvfp4gg.h).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>

#include "gemm.cuh"
#include "gemm_pair.cuh"
#include "gemm_tok_pair.cuh"
#include "gemv.cuh"
#include "nvfp4gg.h"

using namespace nvfp4gg;

// Device error word (one per device that loads the library).
static __device__ int g_error_word;
// Per-expert tile-part counters of the completion-signal entry point
// (epoch-tagged: see epoch_arrive).
static __device__ unsigned long long g_signal_counts[NVFP4GG_MAX_GROUPS];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int status = NVFP4GG_OK;
    int sms = 0;
    int* err = nullptr;          // device address of g_error_word
    bool attr_set[12] = {};      // per kernel variant: max dynamic smem set
    // per kernel variant and cluster size 2..8: 0 not asked yet, 1 a cluster
    // of that many CTAs fits the device, -1 it does not
    int cluster_fits[12][9] = {};
    bool gemv_attr[9] = {};      // per GEMV token count: max dynamic smem set
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
int g_sm_cap = 0;
int g_pair_mode = 2;   // prefill kernel family: 0 single, 1 pairs, 2 automatic, 3 token-major pairs (nvfp4gg.h)
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
unsigned long long g_timeout_ns = 2000000000ull;   // 2 s per device-side wait
// Call numbers for the epoch-tagged arrival counters (split-K, signals).
std::atomic<unsigned long long> g_epoch{0};

int cuda_status(cudaError_t e) { return e == cudaSuccess ? NVFP4GG_OK : NVFP4GG_ERR_CUDA; }

// Per-device one-time set-up: architecture check, SM count, error word.
int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4GG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            return NVFP4GG_ERR_CUDA;
        }
        if (major != 10 || minor != 3) {
            d.status = NVFP4GG_ERR_ARCH;
        } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_error_word) != cudaSuccess) {
            return NVFP4GG_ERR_CUDA;
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn) {
                return NVFP4GG_ERR_CUDA;
            }
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    if (d.status != NVFP4GG_OK) return d.status;
    *out = &d;
    return NVFP4GG_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 3-D u8 tensor map: dims (d0 innermost bytes, d1 rows, d2 groups).
int encode_u8_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz) {
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0, d0 * d1};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NVFP4GG_OK : NVFP4GG_ERR_CUDA;
}

// Token tensor maps, one per tile width 16, 32, ..., tt_max (widths a call
// can use: at most M_max rounded up to 32; the others repeat the 16-row map).
// Encoding costs microseconds per map, so the last few sets are cached by
// (A, A_sf, G, M_max, K, tt_max).
struct TokenMaps {
    const void* A = nullptr;
    const void* A_sf = nullptr;
    int G = 0, M_max = 0, K = 0, tt_max = 0, dev = -1;
    CUtensorMap a[kMaxWidths];
    CUtensorMap asf[kMaxWidths];
};
constexpr int kMapCache = 16;
TokenMaps g_maps[kMapCache];
int g_maps_next = 0;

int token_maps(const void* A, const void* A_sf, int G, int M_max, int K, int tt_max,
               CUtensorMap* out_a, CUtensorMap* out_asf) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4GG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < kMapCache; ++i) {
        const TokenMaps& m = g_maps[i];
        if (m.A == A && m.A_sf == A_sf && m.G == G && m.M_max == M_max && m.K == K &&
            m.tt_max == tt_max && m.dev == dev) {
            std::memcpy(out_a, m.a, sizeof(m.a));
            std::memcpy(out_asf, m.asf, sizeof(m.asf));
            return NVFP4GG_OK;
        }
    }
    TokenMaps& m = g_maps[g_maps_next];
    g_maps_next = (g_maps_next + 1) % kMapCache;
    m.A = nullptr;   // invalid until fully encoded
    const uint64_t kb = (uint64_t)K / 2, ks = (uint64_t)K / 16;
    // widths a call can use: M_max rounded up to 16 (single-CTA tiles) or to
    // 32 (CTA-pair tiles); rows past M_max read as zero
    const int rows_cap = ((M_max + 31) / 32) * 32;
    int rc = NVFP4GG_OK;
    for (int i = 0; i < kMaxWidths; ++i) {
        const uint32_t rows = 16u * (i + 1);
        const uint32_t b = (rows <= (uint32_t)tt_max && rows <= (uint32_t)rows_cap) ? rows : 16u;
        if (i > 0 && b == 16u) {
            m.a[i] = m.a[0];
            m.asf[i] = m.asf[0];
            continue;
        }
        if ((rc = encode_u8_3d(&m.a[i], A, kb, M_max, G, 128, b, CU_TENSOR_MAP_SWIZZLE_128B)) != NVFP4GG_OK ||
            (rc = encode_u8_3d(&m.asf[i], A_sf, ks, M_max, G, 16, b, CU_TENSOR_MAP_SWIZZLE_NONE)) != NVFP4GG_OK)
            return rc;
    }
    m.A_sf = A_sf;
    m.G = G;
    m.M_max = M_max;
    m.K = K;
    m.tt_max = tt_max;
    m.dev = dev;
    m.A = A;
    std::memcpy(out_a, m.a, sizeof(m.a));
    std::memcpy(out_asf, m.asf, sizeof(m.asf));
    return NVFP4GG_OK;
}

int check_gemm_shape(int G, int M_max, int N, int K) {
    if (G < 1 || G > NVFP4GG_MAX_GROUPS) return NVFP4GG_ERR_SHAPE;
    if (M_max < 1 || M_max > (1 << 20)) return NVFP4GG_ERR_SHAPE;
    if (N < NVFP4GG_N_ALIGN || N % NVFP4GG_N_ALIGN != 0 || N > (1 << 20)) return NVFP4GG_ERR_SHAPE;
    if (K < NVFP4GG_K_ALIGN || K % NVFP4GG_K_ALIGN != 0 || K > (1 << 20)) return NVFP4GG_ERR_SHAPE;
    return NVFP4GG_OK;
}

// Decode-sized experts (M_max <= 64): token tiles of at most 32, a deep ring
// for the weight stream.  Larger experts: token tiles of up to 192, so that a
// prefill expert's rows usually fit one tile and its weights stream once, and
// each MMA instruction carries 128 x 192 x 64 (the issuing warp's per-stage
// cost, not the tensor pipe, bounds compute-heavy tiles).
constexpr int kNarrowTT = 32, kNarrowStages = 8;
// decode tiles with K % 512 == 0: stages of two K-tiles (same bytes in flight)
constexpr int kNarrowStages2 = 4;
constexpr int kWideTT = 192, kWideStages = 4;
// Larger experts with N a multiple of 256: CTA pairs (M = 256 per MMA),
// token tiles of up to 192 split 96 + 96 rows, six ring stages.
constexpr int kPairTT = 192, kPairStages = 6;
// Automatic pair mode: CTA pairs for prefill calls up to this M_max (a few
// token tiles per expert: the weight stream dominates and the pair's halved
// token staging and deeper ring pay); compute-heavy experts stay single.
constexpr int kPairAutoMaxRows = 256;
// Token-major pairs: 128 token rows per CTA (one tensor-map box).
constexpr int kTokTT = 128;

// The host fills the maps of every width; a launch carries the NW widths
// from map `first` on.
using GemmParamsAll = GemmParams<kMaxWidths>;

template <int NW>
GemmParams<NW> launch_params(const GemmParamsAll& all, int first) {
    static_assert(NW >= 1 && NW <= kMaxWidths, "map count");
    GemmParams<NW> k;
    std::memset(&k, 0, sizeof(k));
    static_cast<GemmArgs&>(k) = static_cast<const GemmArgs&>(all);
    for (int i = 0; i < NW; ++i) {
        k.tm_a[i] = all.tm_a[first + i];
        k.tm_asf[i] = all.tm_asf[first + i];
    }
    return k;
}

template <int TT, int ST, bool SWIGLU = false, int KSUB = 1>
int launch_variant(DeviceState* d, int slot, const GemmParamsAll& all, cudaStream_t stream) {
    using Cfg = KCfg<TT, ST, KSUB>;
    auto kern = gemm_nt_masked_kernel<TT, ST, SWIGLU, KSUB>;
    if (!d->attr_set[slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
        d->attr_set[slot] = true;
    }
    int grid = d->sms;
    if (g_sm_cap > 0 && g_sm_cap < grid) grid = g_sm_cap;
    GemmParams<TT / 16> k = launch_params<TT / 16>(all, 0);
    if (k.csplit) {
        // split-K in clusters of `split` CTAs: a grid of whole clusters
        const int cs = k.split;
        grid -= grid % cs;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int& fits = d->cluster_fits[slot][cs];
        if (fits == 0) {
            int n = 0;
            fits = (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) ? 1 : -1;
            cudaGetLastError();   // a refused query leaves no sticky error
        }
        if (fits > 0) return cuda_status(cudaLaunchKernelEx(&cfg, kern, k));
        // no room for such clusters: the workspace reduction, else no split
        k.csplit = 0;
        if (!k.ws_part) k.split = 1;
    }
    kern<<<grid, kThreads, Cfg::SMEM_BYTES, stream>>>(k);
    return cuda_status(cudaGetLastError());
}

template <int TT, int ST, bool SWIGLU = false>
int launch_pair_variant(DeviceState* d, int slot, const GemmParamsAll& all, cudaStream_t stream) {
    using Cfg = PairCfg<TT, ST>;
    auto kern = gemm_nt_masked_pair_kernel<TT, ST, SWIGLU>;
    if (!d->attr_set[slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
        d->attr_set[slot] = true;
    }
    int ctas = d->sms;
    if (g_sm_cap > 0 && g_sm_cap < ctas) ctas = g_sm_cap;
    ctas &= ~1;   // whole pairs, never more CTAs than the cap allows
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, launch_params<TT / 16>(all, 0)));
}

// Tensor map of the prepared weight tiles as a 2-D u8 array of 128-byte rows
// (16 KB tiles = 128 rows; the bytes are already swizzled, so the map does not
// swizzle), for the token-major pair kernel's tiled loads.  Cached per buffer.
struct WeightMap {
    const void* B = nullptr;
    uint64_t rows = 0;
    int dev = -1;
    CUtensorMap m;
};
constexpr int kWeightMapCache = 16;
WeightMap g_wmaps[kWeightMapCache];
int g_wmaps_next = 0;

int weight_map(const void* B, uint64_t rows, CUtensorMap* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4GG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < kWeightMapCache; ++i) {
        if (g_wmaps[i].B == B && g_wmaps[i].rows == rows && g_wmaps[i].dev == dev) {
            *out = g_wmaps[i].m;
            return NVFP4GG_OK;
        }
    }
    WeightMap& w = g_wmaps[g_wmaps_next];
    g_wmaps_next = (g_wmaps_next + 1) % kWeightMapCache;
    w.B = nullptr;
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(&w.m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(B), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return NVFP4GG_ERR_CUDA;
    w.rows = rows;
    w.dev = dev;
    w.B = B;
    *out = w.m;
    return NVFP4GG_OK;
}

int launch_tok_pair(DeviceState* d, int slot, const GemmParamsAll& all, const CUtensorMap& tm_w,
                    cudaStream_t stream) {
    // the kernel loads 128-row token boxes only (map index 7)
    const GemmParams<1> p = launch_params<1>(all, kTokTT / 16 - 1);
    using Cfg = TokPairCfg;
    if (!d->attr_set[slot]) {
        if (cudaFuncSetAttribute(gemm_nt_masked_tok_pair_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_LIMIT) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
        d->attr_set[slot] = true;
    }
    int ctas = d->sms;
    if (g_sm_cap > 0 && g_sm_cap < ctas) ctas = g_sm_cap;
    ctas &= ~1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(kTokThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::smem_bytes(p.G);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, gemm_nt_masked_tok_pair_kernel, p, tm_w));
}


}  // namespace

extern "C" {

const char* nvfp4_gg_status_string(int s) {
    switch (s) {
        case NVFP4GG_OK: return "NVFP4GG_OK";
        case NVFP4GG_ERR_NULL: return "NVFP4GG_ERR_NULL: a required pointer is NULL";
        case NVFP4GG_ERR_SHAPE: return "NVFP4GG_ERR_SHAPE: unsupported G, M_max, N or K";
        case NVFP4GG_ERR_ALIGN: return "NVFP4GG_ERR_ALIGN: pointer not aligned as required";
        case NVFP4GG_ERR_ARCH: return "NVFP4GG_ERR_ARCH: device is not compute capability 10.3";
        case NVFP4GG_ERR_CUDA: return "NVFP4GG_ERR_CUDA: a CUDA call failed";
        case NVFP4GG_ERR_TIMEOUT: return "NVFP4GG_ERR_TIMEOUT: a device-side wait ran out";
        case NVFP4GG_ERR_MASK: return "NVFP4GG_ERR_MASK: masked_m outside [0, M_max]";
        case NVFP4GG_ERR_SCRATCH:
            return "NVFP4GG_ERR_SCRATCH: tiles x split_k exceeds NVFP4GG_NOALLOC_MAX_SLOTS";
        default: return "unknown nvfp4gg status";
    }
}

int nvfp4_prepared_weight_bytes(int G, int N, int K, size_t* b_bytes, size_t* sf_bytes) {
    if (!b_bytes || !sf_bytes) return NVFP4GG_ERR_NULL;
    if (G < 1 || G > NVFP4GG_MAX_GROUPS || N < NVFP4GG_N_ALIGN || N % NVFP4GG_N_ALIGN ||
        N > (1 << 20) || K < NVFP4GG_K_ALIGN || K % NVFP4GG_K_ALIGN || K > (1 << 20))
        return NVFP4GG_ERR_SHAPE;
    *b_bytes = (size_t)G * ((N + 127) / 128) * 128 * (K / 2);
    *sf_bytes = (size_t)G * ((N + 127) / 128) * (K / 64) * 512;
    return NVFP4GG_OK;
}

}  // extern "C"

namespace {

// Weight re-layout of the logical weight [G][N][K] held by `codes` /
// `scales`; `swiglu` interleaves gate and up rows (N % 128 == 0).  `ranges`
// are the source buffers' byte ranges, checked against the outputs' (no
// overlap).
struct ByteRange {
    const void* p;
    size_t n;
};

bool overlaps(ByteRange a, ByteRange b) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

int prepare_weights(const WeightSource& codes, const WeightSource& scales, int G, int N, int K,
                    void* B_prep, void* B_sf_prep, void* stream, int swiglu,
                    const ByteRange* ranges, int nranges) {
    if (!codes.src0 || !codes.src1 || !scales.src0 || !scales.src1 || !B_prep || !B_sf_prep)
        return NVFP4GG_ERR_NULL;
    size_t bb = 0, sb = 0;
    int rc = nvfp4_prepared_weight_bytes(G, N, K, &bb, &sb);
    if (rc != NVFP4GG_OK) return rc;
    if (!aligned(codes.src0, 16) || !aligned(codes.src1, 16) || !aligned(scales.src0, 16) ||
        !aligned(scales.src1, 16) || !aligned(B_prep, 16) || !aligned(B_sf_prep, 16))
        return NVFP4GG_ERR_ALIGN;
    const ByteRange outs[2] = {{B_prep, bb}, {B_sf_prep, sb}};
    for (int i = 0; i < nranges; ++i)
        if (overlaps(ranges[i], outs[0]) || overlaps(ranges[i], outs[1])) return NVFP4GG_ERR_SHAPE;
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != NVFP4GG_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int threads = 256;
    const long long cap = 16LL * d->sms;
    long long blocks = ((long long)(bb / 16) + threads - 1) / threads;
    relayout_weight_codes_kernel<<<(int)(blocks < cap ? blocks : cap), threads, 0, st>>>(
        codes, static_cast<uint8_t*>(B_prep), G, N, K, swiglu);
    if (cudaGetLastError() != cudaSuccess) return NVFP4GG_ERR_CUDA;
    blocks = ((long long)(sb / 16) + threads - 1) / threads;
    relayout_weight_scales_kernel<<<(int)(blocks < cap ? blocks : cap), threads, 0, st>>>(
        scales, static_cast<uint8_t*>(B_sf_prep), G, N, K, swiglu);
    return cuda_status(cudaGetLastError());
}

int prepare_single(const void* B, const void* B_sf, int G, int N, int K, void* B_prep,
                   void* B_sf_prep, void* stream, int swiglu) {
    if (!B || !B_sf || !B_prep || !B_sf_prep) return NVFP4GG_ERR_NULL;
    const uint8_t* b = static_cast<const uint8_t*>(B);
    const uint8_t* s = static_cast<const uint8_t*>(B_sf);
    const WeightSource codes{b, b, N, N}, scales{s, s, N, N};
    const ByteRange in[2] = {{B, (size_t)G * N * (K / 2)}, {B_sf, (size_t)G * N * (K / 16)}};
    return prepare_weights(codes, scales, G, N, K, B_prep, B_sf_prep, stream, swiglu, in, 2);
}

}  // namespace

extern "C" {

int nvfp4_prepare_weights(const void* B, const void* B_sf, int G, int N, int K, void* B_prep,
                          void* B_sf_prep, void* stream) {
    return prepare_single(B, B_sf, G, N, K, B_prep, B_sf_prep, stream, 0);
}

int nvfp4_prepare_weights_swiglu(const void* B, const void* B_sf, int G, int N, int K,
                                 void* B_prep, void* B_sf_prep, void* stream) {
    if (N % 128 != 0) return NVFP4GG_ERR_SHAPE;
    return prepare_single(B, B_sf, G, N, K, B_prep, B_sf_prep, stream, 1);
}

int nvfp4_prepare_weights_dual(const void* B1, const void* B1_sf, const void* B2, const void* B2_sf,
                               int G, int N1, int K, int interleave, void* B_prep, void* B_sf_prep,
                               void* stream) {
    if (!B1 || !B1_sf || !B2 || !B2_sf || !B_prep || !B_sf_prep) return NVFP4GG_ERR_NULL;
    if (interleave != 0 && interleave != 1) return NVFP4GG_ERR_SHAPE;
    if (N1 < 1 || N1 > (1 << 19)) return NVFP4GG_ERR_SHAPE;
    const int N = 2 * N1;
    if (check_gemm_shape(G, 1, N, K) != NVFP4GG_OK || N1 % NVFP4GG_N_ALIGN != 0 ||
        (interleave && N % 128 != 0))
        return NVFP4GG_ERR_SHAPE;
    const uint8_t* b1 = static_cast<const uint8_t*>(B1);
    const uint8_t* b2 = static_cast<const uint8_t*>(B2);
    const uint8_t* s1 = static_cast<const uint8_t*>(B1_sf);
    const uint8_t* s2 = static_cast<const uint8_t*>(B2_sf);
    const WeightSource codes{b1, b2, N1, N1}, scales{s1, s2, N1, N1};
    const size_t cb = (size_t)G * N1 * (K / 2), sb = (size_t)G * N1 * (K / 16);
    const ByteRange in[4] = {{B1, cb}, {B2, cb}, {B1_sf, sb}, {B2_sf, sb}};
    return prepare_weights(codes, scales, G, N, K, B_prep, B_sf_prep, stream, interleave, in, 4);
}

}  // extern "C"

namespace {

// Upper bound of the decode kernel's tiles (every expert full) and the
// split-K workspace layout: fp32 partials [tiles][split][32][128], then one
// int counter per tile.
long long decode_tile_bound(int G, int M_max, int N) {
    return (long long)G * ((M_max + kNarrowTT - 1) / kNarrowTT) * ((N + 127) / 128);
}

// Device address of this device's signal counters (looked up once per device).
unsigned long long* g_signal_addr[kMaxDevices] = {};
int signal_counts(unsigned long long** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4GG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_signal_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_signal_counts) != cudaSuccess || !ptr) return NVFP4GG_ERR_CUDA;
        g_signal_addr[dev] = static_cast<unsigned long long*>(ptr);
    }
    *out = g_signal_addr[dev];
    return NVFP4GG_OK;
}

size_t splitk_part_bytes(long long tiles, int split) {
    return (size_t)tiles * split * kNarrowTT * 128 * sizeof(float);
}

// Automatic split: as many ranges as whole sets of the tiles fit the SMs,
// at most 6 (clusters of 8 measured slower than 6) and at least 4 K-tiles
// per range.
int auto_split(DeviceState* d, long long tiles, int K) {
    const int grid = (g_sm_cap > 0 && g_sm_cap < d->sms) ? g_sm_cap : d->sms;
    long long s = tiles > 0 ? grid / tiles : 1;
    if (s > 6) s = 6;
    if (s > K / 1024) s = K / 1024;
    if (s < 1) s = 1;
    return (int)s;
}

int gemm_launch(const void* A, const void* A_sf, const void* B, const void* B_sf, const float* alpha,
                const int* masked_m, void* C, int G, int M_max, int N, int K, int split,
                float* ws_part, unsigned long long* ws_cnt, void* stream, bool swiglu = false,
                int* signals = nullptr, int M_total = 0, uint8_t* qa = nullptr,
                uint8_t* qsf = nullptr, const float* qscale = nullptr) {
    // with the NVFP4 output of the SwiGLU epilogue (qa), C may be null
    if (!A || !A_sf || !B || !B_sf || !alpha || !masked_m || (!C && !qa)) return NVFP4GG_ERR_NULL;
    if (qa && (!qsf || !qscale)) return NVFP4GG_ERR_NULL;
    int rc = check_gemm_shape(G, M_max, N, K);
    if (rc != NVFP4GG_OK) return rc;
    if (!aligned(A, 16) || !aligned(A_sf, 16) || !aligned(B, 16) || !aligned(B_sf, 16) ||
        !aligned(C, 16) || !aligned(alpha, 4) || !aligned(masked_m, 4) || !aligned(qa, 16) ||
        !aligned(qscale, 4))
        return NVFP4GG_ERR_ALIGN;
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != NVFP4GG_OK) return rc;

    const bool narrow = M_max <= 64;
    // a cap of one SM leaves no room for a CTA pair: the single-CTA kernel
    // (same token tile bound, same tensor maps) runs the call instead
    const bool pair_fits = g_sm_cap == 0 || g_sm_cap >= 2;
    const bool pairable = !narrow && !swiglu && !signals && N % 256 == 0 && pair_fits;
    // the SwiGLU epilogue runs on CTA pairs too (not on the token-major
    // ones), in pair modes 1 and 2
    const bool swiglu_pair = !narrow && swiglu && !signals && N % 256 == 0 && pair_fits &&
                             (g_pair_mode == 1 || g_pair_mode == 2);
    // token-major pairs (256 x 256 MMA tiles) for compute-heavy experts
    const bool tok = pairable && M_total == 0 && M_max >= 128 && G <= TokPairCfg::MAX_GROUPS &&
                     (g_pair_mode == 3 || (g_pair_mode == 2 && M_max > kPairAutoMaxRows));
    const bool pair = pairable && !tok &&
                      (g_pair_mode == 1 || (g_pair_mode == 2 && M_max <= kPairAutoMaxRows));
    const int tt_max = narrow ? kNarrowTT : tok ? kTokTT : (pair || swiglu_pair) ? kPairTT : kWideTT;
    GemmParamsAll p;
    std::memset(&p, 0, sizeof(p));
    // packed rows (M_total > 0): one group of M_total rows; else [G][M_max]
    if ((rc = M_total > 0 ? token_maps(A, A_sf, 1, M_total, K, tt_max, p.tm_a, p.tm_asf)
                          : token_maps(A, A_sf, G, M_max, K, tt_max, p.tm_a, p.tm_asf)) != NVFP4GG_OK)
        return rc;
    p.contiguous = M_total > 0 ? 1 : 0;
    p.M_total = M_total;
    p.qa = qa;
    p.qsf = qsf;
    p.qscale = qscale;
    p.wq = static_cast<const uint8_t*>(B);
    p.wsf = static_cast<const uint8_t*>(B_sf);
    p.alpha = alpha;
    p.masked_m = masked_m;
    p.C = static_cast<__nv_bfloat16*>(C);
    p.err = d->err;
    p.G = G;
    p.M_max = M_max;
    p.N = N;
    p.K = K;
    p.NT = (N + 127) / 128;
    p.KS = K / 256;
    p.timeout_ns = g_timeout_ns;
    p.split = 1;
    p.epoch = ++g_epoch;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (narrow && split > 1) {
        const long long tiles = decode_tile_bound(G, M_max, N);
        if (tiles * split >= (1LL << 31)) return NVFP4GG_ERR_SHAPE;
        p.split = split;
        p.ws_part = ws_part;
        p.ws_cnt = ws_cnt;
        // up to 8 ranges (the portable cluster size) reduce within a
        // cluster through distributed shared memory; the workspace is then
        // not touched
        const int grid = (g_sm_cap > 0 && g_sm_cap < d->sms) ? g_sm_cap : d->sms;
        p.csplit = (split <= 8 && !signals && grid >= split) ? 1 : 0;
        if (!p.csplit && !ws_part) p.split = 1;   // no workspace to reduce through
    }
    if (signals) {
        unsigned long long* counts = nullptr;
        if ((rc = signal_counts(&counts)) != NVFP4GG_OK) return rc;
        p.signals = signals;
        p.sig_cnt = counts;
    }
    // decode tiles stream weights from few CTAs when there are few experts:
    // two K-tiles per ring stage where K allows it (split-K ranges are then
    // cut in stages: every range keeps at least one)
    const bool ksub2 = narrow && p.KS % 2 == 0 && p.split * 2 <= p.KS;
    if (swiglu) {
        if (ksub2) return launch_variant<kNarrowTT, kNarrowStages2, true, 2>(d, 7, p, st);
        if (swiglu_pair) return launch_pair_variant<kPairTT, kPairStages, true>(d, 8, p, st);
        return narrow ? launch_variant<kNarrowTT, kNarrowStages, true>(d, 3, p, st)
                      : launch_variant<kWideTT, kWideStages, true>(d, 4, p, st);
    }
    if (ksub2) return launch_variant<kNarrowTT, kNarrowStages2, false, 2>(d, 6, p, st);
    if (narrow) return launch_variant<kNarrowTT, kNarrowStages>(d, 0, p, st);
    if (tok) {
        CUtensorMap tm_w;
        const uint64_t rows = (uint64_t)G * p.NT * p.KS * 128;
        if ((rc = weight_map(B, rows, &tm_w)) != NVFP4GG_OK) return rc;
        return launch_tok_pair(d, 5, p, tm_w, st);
    }
    if (pair) return launch_pair_variant<kPairTT, kPairStages>(d, 2, p, st);
    return launch_variant<kWideTT, kWideStages>(d, 1, p, st);
}

}  // namespace

extern "C" {

int nvfp4_grouped_gemm_nt_masked(const void* A, const void* A_sf, const void* B, const void* B_sf,
                                 const float* alpha, const int* masked_m, void* C, int G, int M_max,
                                 int N, int K, void* stream) {
    // Decode calls with few tiles (at most a quarter of the SMs: one or two
    // experts) and a long K split K over thread-block clusters, so that each
    // tile's weight stream runs on several SMs (measured faster for one
    // expert at N = 2048 and 4096, K = 7168; slower at K = 4096); all other
    // calls run unsplit.  The result is deterministic either way.
    int split = 1;
    DeviceState* d = nullptr;
    if (M_max <= 64 && K >= 24 * 256 && check_gemm_shape(G, M_max, N, K) == NVFP4GG_OK &&
        device_state(&d) == NVFP4GG_OK) {
        const long long tiles = decode_tile_bound(G, M_max, N);
        const int grid = (g_sm_cap > 0 && g_sm_cap < d->sms) ? g_sm_cap : d->sms;
        if (tiles * 4 <= grid) split = auto_split(d, tiles, K);
    }
    return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, split, nullptr,
                       nullptr, stream);
}

}  // extern "C"

namespace {

template <int M>
int launch_gemv(DeviceState* d, const void* x, const void* B, const void* B_sf, const float* alpha,
                void* y, int N, int K, cudaStream_t st) {
    constexpr int R = M <= 4 ? 2 : 1;   // weight rows per warp (register budget, grid balance)
    auto kern = gemv_w4a16_kernel<M, R>;
    const int smem = (int)gemv_smem_bytes(M, K);
    if (!d->gemv_attr[M]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kGemvMaxSmem) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
        d->gemv_attr[M] = true;
    }
    // as many CTAs per SM as registers and the staged tokens allow, groups of
    // R rows grid-strided over all warps
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGemvThreads, smem) !=
            cudaSuccess || per_sm < 1)
        per_sm = 1;
    const long long need = (((long long)N + R - 1) / R * 32 + kGemvThreads - 1) / kGemvThreads;
    long long grid = (long long)per_sm * d->sms;
    if (grid > need) grid = need;
    kern<<<(int)grid, kGemvThreads, smem, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const uint8_t*>(B),
        static_cast<const uint8_t*>(B_sf), alpha, static_cast<__nv_bfloat16*>(y), N, K);
    return cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" {

int nvfp4_gemv_w4a16(const void* x, const void* B, const void* B_sf, const float* alpha, void* y,
                     int M, int N, int K, void* stream) {
    if (!x || !B || !B_sf || !alpha || !y) return NVFP4GG_ERR_NULL;
    if (M < 1 || M > kGemvMaxTokens || N < 1 || N > (1 << 24) || K < 32 || K % 32 != 0 ||
        gemv_smem_bytes(M, K) > kGemvMaxSmem)
        return NVFP4GG_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(B, 16) || !aligned(B_sf, 2) || !aligned(y, 2) ||
        !aligned(alpha, 4))
        return NVFP4GG_ERR_ALIGN;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != NVFP4GG_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (M) {
        case 1: return launch_gemv<1>(d, x, B, B_sf, alpha, y, N, K, st);
        case 2: return launch_gemv<2>(d, x, B, B_sf, alpha, y, N, K, st);
        case 3: return launch_gemv<3>(d, x, B, B_sf, alpha, y, N, K, st);
        case 4: return launch_gemv<4>(d, x, B, B_sf, alpha, y, N, K, st);
        case 5: return launch_gemv<5>(d, x, B, B_sf, alpha, y, N, K, st);
        case 6: return launch_gemv<6>(d, x, B, B_sf, alpha, y, N, K, st);
        case 7: return launch_gemv<7>(d, x, B, B_sf, alpha, y, N, K, st);
        default: return launch_gemv<8>(d, x, B, B_sf, alpha, y, N, K, st);
    }
}

int nvfp4_grouped_gemm_nt_contiguous(const void* A, const void* A_sf, const void* B,
                                     const void* B_sf, const float* alpha, const int* masked_m,
                                     void* C, int G, int M_max, int M_total, int N, int K,
                                     void* stream) {
    if (M_total < 1 || M_total > (1 << 24) || M_max > M_total) return NVFP4GG_ERR_SHAPE;
    return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, 1, nullptr, nullptr,
                       stream, false, nullptr, M_total);
}

int nvfp4_grouped_gemm_nt_masked_signals(const void* A, const void* A_sf, const void* B,
                                         const void* B_sf, const float* alpha, const int* masked_m,
                                         void* C, int G, int M_max, int N, int K, int* dst_signals,
                                         void* stream) {
    if (!dst_signals) return NVFP4GG_ERR_NULL;
    if (!aligned(dst_signals, 4)) return NVFP4GG_ERR_ALIGN;
    return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, 1, nullptr, nullptr,
                       stream, false, dst_signals);
}

int nvfp4_grouped_gemm_nt_masked_swiglu(const void* A, const void* A_sf, const void* B,
                                        const void* B_sf, const float* alpha, const int* masked_m,
                                        void* C, int G, int M_max, int N, int K, void* stream) {
    if (N % 128 != 0) return NVFP4GG_ERR_SHAPE;
    return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, 1, nullptr, nullptr,
                       stream, true);
}

int nvfp4_grouped_gemm_nt_masked_swiglu_quant(const void* A, const void* A_sf, const void* B,
                                              const void* B_sf, const float* alpha,
                                              const int* masked_m, void* C, const float* qscale,
                                              void* A2, void* A2_sf, int G, int M_max, int N, int K,
                                              void* stream) {
    if (!A2 || !A2_sf || !qscale) return NVFP4GG_ERR_NULL;
    if (N % 128 != 0) return NVFP4GG_ERR_SHAPE;
    return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, 1, nullptr, nullptr,
                       stream, true, nullptr, 0, static_cast<uint8_t*>(A2),
                       static_cast<uint8_t*>(A2_sf), qscale);
}

int nvfp4_quantize_bf16(const void* x, const float* qscale, void* codes, void* sf, int R, int L,
                        int rows_per_scale, void* stream) {
    if (!x || !qscale || !codes || !sf) return NVFP4GG_ERR_NULL;
    if (R < 1 || L < 16 || L % 16 != 0 || rows_per_scale < 1 || (long long)R * L > (1LL << 40))
        return NVFP4GG_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(codes, 8) || !aligned(qscale, 4)) return NVFP4GG_ERR_ALIGN;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != NVFP4GG_OK) return rc;
    const long long blocks = (long long)R * (L / 16);
    long long grid = (blocks + 255) / 256;
    const long long cap = (long long)d->sms * 8;   // grid-stride beyond 8 CTAs per SM
    if (grid > cap) grid = cap;
    quantize_bf16_kernel<<<(int)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(x), qscale, static_cast<uint8_t*>(codes),
        static_cast<uint8_t*>(sf), blocks, L, rows_per_scale);
    return cuda_status(cudaGetLastError());
}

size_t nvfp4_splitk_workspace_bytes(int G, int M_max, int N, int K, int split_k) {
    if (check_gemm_shape(G, M_max, N, K) != NVFP4GG_OK || split_k < 0 || split_k > 16) return 0;
    if (M_max > 64) return 16;   // prefill shapes run unsplit: no workspace needed
    const long long tiles = decode_tile_bound(G, M_max, N);
    const int s = split_k == 0 ? 16 : split_k;
    return ((splitk_part_bytes(tiles, s) + 255) & ~(size_t)255) + (size_t)tiles * 8;
}

int nvfp4_grouped_gemm_nt_masked_splitk(const void* A, const void* A_sf, const void* B,
                                        const void* B_sf, const float* alpha, const int* masked_m,
                                        void* C, int G, int M_max, int N, int K, int split_k,
                                        void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace) return NVFP4GG_ERR_NULL;
    if (split_k < 0 || split_k > 16) return NVFP4GG_ERR_SHAPE;
    int rc = check_gemm_shape(G, M_max, N, K);
    if (rc != NVFP4GG_OK) return rc;
    if (!aligned(workspace, 256)) return NVFP4GG_ERR_ALIGN;
    if (M_max > 64)
        return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, 1, nullptr,
                           nullptr, stream);
    int split = split_k;
    if (split == 0) {
        DeviceState* d = nullptr;
        if ((rc = device_state(&d)) != NVFP4GG_OK) return rc;
        split = auto_split(d, decode_tile_bound(G, M_max, N), K);
    }
    if (split > K / 256) split = K / 256;
    if (split < 1) split = 1;
    const long long tiles = decode_tile_bound(G, M_max, N);
    const size_t part = (splitk_part_bytes(tiles, split) + 255) & ~(size_t)255;
    if (workspace_bytes < part + (size_t)tiles * 8) return NVFP4GG_ERR_SHAPE;
    float* ws_part = static_cast<float*>(workspace);
    unsigned long long* ws_cnt =
        reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) + part);
    return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, split, ws_part, ws_cnt,
                       stream);
}

}  // extern "C"

namespace {

// Address under which the current device reaches host buffer `h`: pinned
// (page-locked) host memory is mapped into the device's address space;
// pageable memory is not (nullptr).
void* host_mapped(const void* h) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
    return a.devicePointer;
}

// The host-buffer entry copies large activations in expert chunks on a side
// stream, so that later chunks cross the CPU-GPU link while earlier chunks'
// GEMMs run (measured on GB300: host-to-device copies and the GEMM's stores
// into host memory share the link only in part).  The chunks grow fourfold
// (experts in the ratio 1 : 4 : 16 : 64): the first copy, which nothing
// hides, stays short, and each further copy still ends before the previous
// chunk's GEMM, whose output is several times its input in every prefill
// shape.  Per device: the side stream, an event marking the caller's stream
// at entry, and one event per chunk that the chunk's GEMM waits for.
// Created on first use; nvfp4_gg_shutdown forgets them (after a device
// reset they are gone with the context).
constexpr int kHostChunks = 4;
struct HostPipe {
    bool ready = false;
    cudaStream_t copy = nullptr;
    cudaEvent_t entry = nullptr;
    cudaEvent_t chunk[kHostChunks] = {};
};
std::mutex g_host_mu;   // held over a call's whole enqueue; taken before g_mu, never after it
HostPipe g_pipe[kMaxDevices];

// The current device's pipe; the caller holds g_host_mu.
int host_pipe(HostPipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4GG_ERR_CUDA;
    HostPipe& hp = g_pipe[dev];
    if (!hp.ready) {
        if (cudaStreamCreateWithFlags(&hp.copy, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.entry, cudaEventDisableTiming) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
        for (int j = 0; j < kHostChunks; ++j)
            if (cudaEventCreateWithFlags(&hp.chunk[j], cudaEventDisableTiming) != cudaSuccess)
                return NVFP4GG_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return NVFP4GG_OK;
}

// Expert chunks of the host-buffer entry: end[j] is one past chunk j's last
// expert; returns the number of chunks.  One chunk unless the call has
// prefill-sized experts (M_max > 64: the plain entry never splits K there,
// so every chunk runs the kernel the whole call would) and at least 2 MiB of
// activations; two from 2 MiB, three from 8 MiB, four from 32 MiB, never
// more than G.  Chunk j holds about G 4^j / (1 + 4 + ... + 4^(P-1))
// experts, at least one.
int host_chunks(int G, int M_max, size_t in_bytes, int* end) {
    int P = 1;
    if (M_max > 64 && G <= TokPairCfg::MAX_GROUPS)
        P = in_bytes >= (32u << 20) ? 4 : in_bytes >= (8u << 20) ? 3 : in_bytes >= (2u << 20) ? 2 : 1;
    if (P > G) P = G;
    const long long total = ((1LL << (2 * P)) - 1) / 3;   // 1 + 4 + ... + 4^(P-1)
    long long cum = 0;
    int prev = 0;
    for (int j = 0; j < P; ++j) {
        cum += 1LL << (2 * j);
        int e = (int)((G * cum + total / 2) / total);
        if (e < prev + 1) e = prev + 1;
        if (e > G - (P - 1 - j)) e = G - (P - 1 - j);
        end[j] = prev = e;
    }
    return P;
}

}  // namespace

extern "C" {

size_t nvfp4_host_staging_bytes(int G, int M_max, int N, int K) {
    if (check_gemm_shape(G, M_max, N, K) != NVFP4GG_OK) return 0;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return up((size_t)G * M_max * N * 2) + up((size_t)G * M_max * (K / 2)) +
           up((size_t)G * M_max * (K / 16)) + up((size_t)G * 4) + up((size_t)G * 4);
}

int nvfp4_grouped_gemm_nt_masked_host(const void* h_A, const void* h_A_sf, const float* h_alpha,
                                      const int* h_masked_m, const void* B, const void* B_sf,
                                      void* h_C, int G, int M_max, int N, int K, void* d_staging,
                                      size_t staging_bytes, void* stream) {
    if (!h_A || !h_A_sf || !h_alpha || !h_masked_m || !B || !B_sf || !h_C || !d_staging)
        return NVFP4GG_ERR_NULL;
    int rc = check_gemm_shape(G, M_max, N, K);
    if (rc != NVFP4GG_OK) return rc;
    if (staging_bytes < nvfp4_host_staging_bytes(G, M_max, N, K)) return NVFP4GG_ERR_SHAPE;
    if (!aligned(d_staging, 16)) return NVFP4GG_ERR_ALIGN;
    for (int g = 0; g < G; ++g)
        if (h_masked_m[g] < 0 || h_masked_m[g] > M_max) return NVFP4GG_ERR_SHAPE;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t c_bytes = (size_t)G * M_max * N * 2;
    const size_t a_bytes = (size_t)G * M_max * (K / 2);
    const size_t asf_bytes = (size_t)G * M_max * (K / 16);
    uint8_t* dC = static_cast<uint8_t*>(d_staging);
    uint8_t* dA = dC + up(c_bytes);
    uint8_t* dAsf = dA + up(a_bytes);
    float* dAlpha = reinterpret_cast<float*>(dAsf + up(asf_bytes));
    int* dMask = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(dAlpha) + up((size_t)G * 4));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Pinned host buffers are used in place: the kernel reads alpha and
    // masked_m and its epilogue writes the valid rows of C over the CPU-GPU
    // link, saving a copy (about 10 us of latency each) per buffer and per
    // non-empty expert.  The activations are always copied: the kernel reads
    // each token tile once per weight block.
    const float* alpha_in = static_cast<const float*>(host_mapped(h_alpha));
    const int* mask_in = static_cast<const int*>(host_mapped(h_masked_m));
    void* c_out = host_mapped(h_C);
    if (c_out && !aligned(c_out, 16)) c_out = nullptr;
    const size_t group_bytes = (size_t)M_max * N * 2;
    int chunk_end[kHostChunks];
    const int P = host_chunks(G, M_max, a_bytes + asf_bytes, chunk_end);
    std::unique_lock<std::mutex> pipe_lock(g_host_mu, std::defer_lock);
    HostPipe* hp = nullptr;
    if (P > 1) {
        pipe_lock.lock();
        if ((rc = host_pipe(&hp)) != NVFP4GG_OK) return rc;
        // the side stream's copies may overwrite the staging buffer only
        // after the work queued on `stream` before this call (a previous
        // call's GEMM still reading it)
        if (cudaEventRecord(hp->entry, st) != cudaSuccess ||
            cudaStreamWaitEvent(hp->copy, hp->entry, 0) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
    } else if (cudaMemcpyAsync(dA, h_A, a_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess ||
               cudaMemcpyAsync(dAsf, h_A_sf, asf_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) {
        return NVFP4GG_ERR_CUDA;
    }
    if (!alpha_in) {
        if (cudaMemcpyAsync(dAlpha, h_alpha, (size_t)G * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
        alpha_in = dAlpha;
    }
    if (!mask_in) {
        if (cudaMemcpyAsync(dMask, h_masked_m, (size_t)G * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
        mask_in = dMask;
    }
    uint8_t* c_dst = static_cast<uint8_t*>(c_out ? c_out : dC);
    if (P == 1) {
        rc = nvfp4_grouped_gemm_nt_masked(dA, dAsf, B, B_sf, alpha_in, mask_in, c_dst, G, M_max, N,
                                          K, stream);
    } else {
        // chunk j: its experts' rows of A and A_sf copied on the side
        // stream, its GEMM on `stream` after that copy
        size_t b_expert = 0, sf_expert = 0;
        if ((rc = nvfp4_prepared_weight_bytes(1, N, K, &b_expert, &sf_expert)) != NVFP4GG_OK)
            return rc;
        const size_t a_row = (size_t)K / 2, sf_row = (size_t)K / 16;
        for (int j = 0; j < P && rc == NVFP4GG_OK; ++j) {
            const int g0 = j == 0 ? 0 : chunk_end[j - 1];
            const int g1 = chunk_end[j];
            const size_t r0 = (size_t)g0 * M_max, nr = (size_t)(g1 - g0) * M_max;
            if (cudaMemcpyAsync(dA + r0 * a_row, static_cast<const uint8_t*>(h_A) + r0 * a_row,
                                nr * a_row, cudaMemcpyHostToDevice, hp->copy) != cudaSuccess ||
                cudaMemcpyAsync(dAsf + r0 * sf_row, static_cast<const uint8_t*>(h_A_sf) + r0 * sf_row,
                                nr * sf_row, cudaMemcpyHostToDevice, hp->copy) != cudaSuccess ||
                cudaEventRecord(hp->chunk[j], hp->copy) != cudaSuccess ||
                cudaStreamWaitEvent(st, hp->chunk[j], 0) != cudaSuccess)
                return NVFP4GG_ERR_CUDA;
            rc = nvfp4_grouped_gemm_nt_masked(
                dA + r0 * a_row, dAsf + r0 * sf_row, static_cast<const uint8_t*>(B) + g0 * b_expert,
                static_cast<const uint8_t*>(B_sf) + g0 * sf_expert, alpha_in + g0, mask_in + g0,
                c_dst + g0 * group_bytes, g1 - g0, M_max, N, K, stream);
        }
    }
    if (rc != NVFP4GG_OK || c_out) return rc;
    for (int g = 0; g < G; ++g) {
        if (h_masked_m[g] == 0) continue;
        if (cudaMemcpyAsync(static_cast<uint8_t*>(h_C) + g * group_bytes, dC + g * group_bytes,
                            (size_t)h_masked_m[g] * N * 2, cudaMemcpyDeviceToHost, st) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
    }
    return NVFP4GG_OK;
}

int nvfp4_gg_set_sm_count(int sm_count) {
    if (sm_count < 0) return NVFP4GG_ERR_SHAPE;
    std::lock_guard<std::mutex> lock(g_mu);
    g_sm_cap = sm_count;
    return NVFP4GG_OK;
}

int nvfp4_gg_set_pair_mode(int mode) {
    if (mode < 0 || mode > 3) return NVFP4GG_ERR_SHAPE;
    std::lock_guard<std::mutex> lock(g_mu);
    g_pair_mode = mode;
    return NVFP4GG_OK;
}

int nvfp4_gg_check_error(void* stream) {
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != NVFP4GG_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return NVFP4GG_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, d->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return NVFP4GG_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(d->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return NVFP4GG_ERR_CUDA;
    }
    return word;
}

int nvfp4_gg_selftest_watchdog(long long timeout_ns, void* stream) {
    if (timeout_ns < 1000 || timeout_ns > 10000000000LL) return NVFP4GG_ERR_SHAPE;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != NVFP4GG_OK) return rc;
    watchdog_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        d->err, (unsigned long long)timeout_ns);
    return cuda_status(cudaGetLastError());
}

int nvfp4_gg_mma_peak_probe(int iters, int n, int ctas, void* stream) {
    if (iters < 1 || iters > (1 << 24) || n < 16 || n > 256 || n % 16 != 0 || ctas < 0)
        return NVFP4GG_ERR_SHAPE;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != NVFP4GG_OK) return rc;
    constexpr int kSmem = 51216 + 1024;
    if (cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess)
        return NVFP4GG_ERR_CUDA;
    const int grid = (ctas == 0 || ctas > d->sms) ? d->sms : ctas;
    mma_peak_kernel<<<grid, 128, kSmem, static_cast<cudaStream_t>(stream)>>>(iters, n, d->err,
                                                                             g_timeout_ns);
    return cuda_status(cudaGetLastError());
}

int nvfp4_gg_mma_peak_probe_pair(int iters, int n, int clusters, void* stream) {
    if (iters < 1 || iters > (1 << 24) || n < 16 || n > 256 || n % 16 != 0 || clusters < 0)
        return NVFP4GG_ERR_SHAPE;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != NVFP4GG_OK) return rc;
    // operands use 33 KB; asking for more than half an SM's shared memory
    // keeps every CTA of the probe on an SM of its own (no CTA waits in
    // tcgen05.alloc for a CTA of another cluster)
    constexpr int kSmem = 120 * 1024;
    if (cudaFuncSetAttribute(mma_peak_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem) != cudaSuccess)
        return NVFP4GG_ERR_CUDA;
    const int max_clusters = d->sms / 2;
    const int ncl = (clusters == 0 || clusters > max_clusters) ? max_clusters : clusters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * ncl, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, mma_peak_pair_kernel, iters, n, d->err, g_timeout_ns));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Split-K with a library-owned scratch (nvfp4_grouped_gemm_nt_masked_splitk_noalloc).
// The scratch is a static device array, laid out like a caller workspace:
// fp32 partials for NVFP4GG_NOALLOC_MAX_SLOTS (tile, K-range) slots, then one
// int arrival counter per slot.  Every device that loads the module gets its
// own copy, zero-initialised.

namespace {

constexpr size_t kNoAllocPartBytes =
    (size_t)NVFP4GG_NOALLOC_MAX_SLOTS * kNarrowTT * 128 * sizeof(float);   // 4 MiB
constexpr size_t kNoAllocBytes = kNoAllocPartBytes + NVFP4GG_NOALLOC_MAX_SLOTS * 8;
static_assert(kNoAllocPartBytes % 256 == 0, "counters must start 256-byte aligned");

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

unsigned char* g_noalloc_addr[kMaxDevices] = {};

// Device address of this device's scratch, looked up on the first call made
// with the device current.
int noalloc_scratch(unsigned char** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4GG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return NVFP4GG_ERR_CUDA;
        g_noalloc_addr[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_noalloc_addr[dev];
    return NVFP4GG_OK;
}

}  // namespace

extern "C" int nvfp4_grouped_gemm_nt_masked_splitk_noalloc(
    const void* A, const void* A_sf, const void* B, const void* B_sf, const float* alpha,
    const int* masked_m, void* C, int G, int M_max, int N, int K, int split_k, void* stream) {
    if (!A || !A_sf || !B || !B_sf || !alpha || !masked_m || !C) return NVFP4GG_ERR_NULL;
    if (split_k < 0 || split_k > 16) return NVFP4GG_ERR_SHAPE;
    int rc = check_gemm_shape(G, M_max, N, K);
    if (rc != NVFP4GG_OK) return rc;
    if (M_max > 64 || split_k == 1)
        return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, 1, nullptr,
                           nullptr, stream);
    const long long tiles = decode_tile_bound(G, M_max, N);
    const long long slots = NVFP4GG_NOALLOC_MAX_SLOTS;
    int split = split_k;
    if (split > K / 256) split = K / 256;
    if (split_k > 1 && split > 1 && tiles * split > slots) return NVFP4GG_ERR_SCRATCH;
    if (split_k == 0) {
        DeviceState* d = nullptr;
        if ((rc = device_state(&d)) != NVFP4GG_OK) return rc;
        split = auto_split(d, tiles, K);
        // auto_split keeps tiles x split <= SMs, below the slot count on
        // every GPU with at most NVFP4GG_NOALLOC_MAX_SLOTS SMs (GB300: 152),
        // so this guard only acts on larger GPUs
        if (tiles * split > slots) split = (int)(slots / tiles);
    }
    if (split <= 1)
        return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, 1, nullptr,
                           nullptr, stream);
    unsigned char* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != NVFP4GG_OK) return rc;
    return gemm_launch(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K, split,
                       reinterpret_cast<float*>(scratch),
                       reinterpret_cast<unsigned long long*>(scratch + kNoAllocPartBytes), stream);
}

// ---------------------------------------------------------------------------
// Dropping the host-side caches (every other file-scope cache is above).

extern "C" {

int nvfp4_gg_shutdown(void) {
    std::lock_guard<std::mutex> pipe_lock(g_host_mu);
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < kMaxDevices; ++i) {
        g_dev[i] = DeviceState{};
        g_pipe[i] = HostPipe{};
        g_signal_addr[i] = nullptr;
        g_noalloc_addr[i] = nullptr;
    }
    for (int i = 0; i < kMapCache; ++i) g_maps[i].A = nullptr;
    for (int i = 0; i < kWeightMapCache; ++i) g_wmaps[i].B = nullptr;
    return NVFP4GG_OK;
}

}  // extern "C"
