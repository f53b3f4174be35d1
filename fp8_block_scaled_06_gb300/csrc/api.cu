// C ABI of the FP8 GEMM library: argument checks, TMA tensor-map encoding
// (cached), per-device status word, scale packing temporaries, kernel choice
// and launch.
//
// TMA rules checked on the host before any launch (Triton tutorial ch. 12,
// 12.2.3): base address 16-byte aligned, innermost stride 1, every other
// stride a multiple of 16 bytes, 2-5 dimensions.  Tensor maps are encoded once
// per (pointer, shape, box) and reused ("create the descriptor outside the
// loop", 12.8 Q1 of the same chapter).
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "internal.h"

namespace fp8g {

// Per-device status word: [0] first error code since the last read, [1] detail.
__device__ unsigned int g_status_word[2];

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
unsigned int *g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
bool g_dev_ok[kMaxDevices] = {};
std::atomic<uint64_t> g_timeout_ns{0};

uint64_t timeout_ns() {
    uint64_t t = g_timeout_ns.load(std::memory_order_relaxed);
    if (t == 0) {
        uint64_t ms = 2000;
        if (const char *env = std::getenv("FP8G_WAIT_TIMEOUT_MS")) {
            const long long v = std::atoll(env);
            if (v > 0) ms = (uint64_t)v;
        }
        t = ms * 1000000ull;
        g_timeout_ns.store(t, std::memory_order_relaxed);
    }
    return t;
}

cudaMemPool_t g_pool[kMaxDevices] = {};
bool g_pool_ok[kMaxDevices] = {};

// Library-owned device memory pool for the packed scale temporaries: memory
// returned with cudaFreeAsync stays in the pool (release threshold = max), so
// steady-state calls do not touch the driver allocator.
fp8g_status scale_pool(int dev, cudaMemPool_t &pool) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_pool_ok[dev]) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if (cudaMemPoolCreate(&g_pool[dev], &props) != cudaSuccess) return FP8G_ERR_CUDA;
        uint64_t thr = ~0ull;
        cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold, &thr);
        g_pool_ok[dev] = true;
    }
    pool = g_pool[dev];
    return FP8G_OK;
}

struct DevInfo {
    int dev;
    int num_sms;
    unsigned int *status;
};

fp8g_status device_info(DevInfo &di) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8G_ERR_DEVICE;
    if (dev < 0 || dev >= kMaxDevices) return FP8G_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev_ok[dev]) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FP8G_ERR_DEVICE;
        if (major != 10 || minor != 3) return FP8G_ERR_DEVICE;  // built for sm_103a only
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return FP8G_ERR_CUDA;
        if (g_encode == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return FP8G_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
        g_num_sms[dev] = sms;
        g_dev_ok[dev] = true;
    }
    di.dev = dev;
    di.num_sms = g_num_sms[dev];
    di.status = g_status_ptr[dev];
    return FP8G_OK;
}

// ------------------------------------------------------------ tensor maps
struct TmapKey {
    const void *ptr;
    int rank, dtype, ebits, swizzle, dev;
    uint64_t dims[3];
    uint32_t box[3];
    bool operator==(const TmapKey &o) const {
        return ptr == o.ptr && rank == o.rank && dtype == o.dtype && ebits == o.ebits &&
               swizzle == o.swizzle && dev == o.dev && std::memcmp(dims, o.dims, sizeof dims) == 0 &&
               std::memcmp(box, o.box, sizeof box) == 0;
    }
};

struct TmapKeyHash {
    size_t operator()(const TmapKey &k) const {
        uint64_t h = 1469598103934665603ull;  // FNV-1a over the fields
        auto mix = [&h](uint64_t v) {
            for (int i = 0; i < 8; ++i) {
                h ^= (v >> (8 * i)) & 0xFFu;
                h *= 1099511628211ull;
            }
        };
        mix(reinterpret_cast<uintptr_t>(k.ptr));
        mix(((uint64_t)k.rank << 48) ^ ((uint64_t)k.dtype << 32) ^ ((uint64_t)k.ebits << 16) ^
            ((uint64_t)k.swizzle << 8) ^ (uint64_t)k.dev);
        for (int i = 0; i < 3; ++i) mix(k.dims[i] ^ ((uint64_t)k.box[i] << 40));
        return (size_t)h;
    }
};

// Encoded maps by key; cleared when it reaches kCacheMax entries (a process
// that keeps creating new operand buffers does not grow it without bound).
constexpr size_t kCacheMax = 4096;
std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> g_cache;

// Dense row-major tensor [dims[rank-1]] ... [dims[0]] (dims[0] innermost,
// contiguous), element size ebits bits, zero fill out of bounds.
fp8g_status tmap_encode(const void *ptr, CUtensorMapDataType dtype, int ebits, int rank,
                        const uint64_t *dims, const uint32_t *box, CUtensorMapSwizzle swz, int dev,
                        CUtensorMap &out) {
    TmapKey key{};
    key.ptr = ptr;
    key.rank = rank;
    key.dtype = (int)dtype;
    key.ebits = ebits;
    key.swizzle = (int)swz;
    key.dev = dev;
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
    }
    std::lock_guard<std::mutex> lk(g_mu);
    const auto it = g_cache.find(key);
    if (it != g_cache.end()) {
        out = it->second;
        return FP8G_OK;
    }
    cuuint64_t gdim[3], gstride[2];
    cuuint32_t bdim[3], estr[3];
    uint64_t stride_bits = (uint64_t)ebits;
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estr[i] = 1;
        if (i > 0) gstride[i - 1] = stride_bits / 8;
        stride_bits *= dims[i];
    }
    CUtensorMap m;
    const CUresult r = g_encode(&m, dtype, (cuuint32_t)rank, const_cast<void *>(ptr), gdim, gstride,
                                bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return FP8G_ERR_CUDA;
    if (g_cache.size() >= kCacheMax) g_cache.clear();
    g_cache.emplace(key, m);
    out = m;
    return FP8G_OK;
}

// Operand tile map, 128-byte swizzle (the tcgen05 K-major SW128 layout).
// dims / box count elements.  FP8: one byte per element in memory and in
// shared memory.  E2M1: two codes per byte in memory (the first in the low
// nibble); the 16U4_ALIGN16B load widens every 16 codes (8 bytes) to a
// 16-byte slot of shared memory, the 8 data bytes followed by 8 unused ones,
// which is how kind::f8f6f4 / mxf8f6f4 MMAs read 4-bit operands, so a tile
// takes the same shared memory as an FP8 tile of the same shape; the load
// counts only the packed bytes (half of that) toward the stage's mbarrier.
// FP6 (E2M3, E3M2): four codes per three bytes in memory; the 16U6_ALIGN16B
// load widens every 16 codes (12 bytes) to a 16-byte slot (4 unused bytes)
// and counts three quarters of the tile.
fp8g_status tmap_operand(const void *ptr, int fmt, int rank, const uint64_t *dims,
                         const uint32_t *box, int dev, CUtensorMap &out) {
    if (fmt == FP8G_E2M1)
        return tmap_encode(ptr, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, rank, dims, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, dev, out);
    if (fmt == FP8G_E2M3 || fmt == FP8G_E3M2)
        return tmap_encode(ptr, CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B, 6, rank, dims, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, dev, out);
    return tmap_encode(ptr, CU_TENSOR_MAP_DATA_TYPE_UINT8, 8, rank, dims, box,
                       CU_TENSOR_MAP_SWIZZLE_128B, dev, out);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_fmt(int f) { return f >= FP8G_E4M3 && f <= FP8G_E3M2; }

// The MMA instruction descriptor's A / B type field (kind::f8f6f4 and
// kind::mxf8f6f4): E4M3 0, E5M2 1, E2M3 3, E3M2 4, E2M1 5.
uint32_t mma_type(int f) { return f == FP8G_E2M1 ? 5u : (uint32_t)f; }

// Packed operands (E2M1, FP6)
bool packed_fmt(int f) { return f == FP8G_E2M1 || f == FP8G_E2M3 || f == FP8G_E3M2; }

// Eighths of an operand tile that its packed load does not deliver.
int32_t gap8(int f) { return f == FP8G_E2M1 ? 4 : (f == FP8G_E2M3 || f == FP8G_E3M2) ? 2 : 0; }

// Packed operands: the 16U4 / 16U6 tile maps want K a multiple of 128 and the
// operand's base 32-byte aligned (its row stride, K / 2 or 3K / 4 bytes, is
// then a multiple of 32).
fp8g_status check_packed(const void *A, const void *B, int a_fmt, int b_fmt, int64_t K) {
    if (!packed_fmt(a_fmt) && !packed_fmt(b_fmt)) return FP8G_OK;
    if (K % 128 != 0) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if ((packed_fmt(a_fmt) && !aligned(A, 32)) || (packed_fmt(b_fmt) && !aligned(B, 32)))
        return FP8G_ERR_ALIGNMENT;
    return FP8G_OK;
}

constexpr int64_t kMaxDim = (int64_t)1 << 31;

// Shape / alignment rules common to every GEMM entry point.
fp8g_status check_common(const void *A, const void *B, const void *C, int out, int64_t M,
                         int64_t N, int64_t K) {
    if (A == nullptr || B == nullptr || C == nullptr) return FP8G_ERR_INVALID_ARG;
    if (out != FP8G_OUT_BF16 && out != FP8G_OUT_F32) return FP8G_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return FP8G_ERR_INVALID_ARG;
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return FP8G_ERR_ALIGNMENT;
    if (K % 16 != 0) return FP8G_ERR_ALIGNMENT;
    const int64_t esz = out == FP8G_OUT_F32 ? 4 : 2;
    if ((N * esz) % 16 != 0) return FP8G_ERR_ALIGNMENT;
    return FP8G_OK;
}

// Argument rules of the grouped GEMM (fp8_grouped_gemm_scatter and the
// entry points built on it), checked on the host before any launch.
fp8g_status check_grouped_args(const void *A, const void *B, const float *sfa, const float *sfb,
                                const void *C, int out, const int32_t *counts, int32_t E,
                                int64_t N, int64_t K, int64_t total_rows,
                                const int32_t *c_row_of, int64_t c_rows,
                                const int32_t *offsets_out, const int32_t *tile_map_out) {
    if (c_row_of != nullptr && (!aligned(c_row_of, 4) || c_rows < 1)) return FP8G_ERR_INVALID_ARG;
    if (c_row_of != nullptr && c_rows >= kMaxDim) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (counts == nullptr || sfa == nullptr || sfb == nullptr) return FP8G_ERR_INVALID_ARG;
    if (E < 1) return FP8G_ERR_INVALID_ARG;
    if (E > FP8G_MAX_EXPERTS) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (total_rows < 0) return FP8G_ERR_INVALID_ARG;
    if (total_rows > 0) {
        fp8g_status st = check_common(A, B, C, out, total_rows, N, K);
        if (st != FP8G_OK) return st;
    } else {
        if (B == nullptr) return FP8G_ERR_INVALID_ARG;
        if (out != FP8G_OUT_BF16 && out != FP8G_OUT_F32) return FP8G_ERR_INVALID_ARG;
        if (N < 1 || K < 1) return FP8G_ERR_INVALID_ARG;
        if (!aligned(B, 16) || K % 16 != 0) return FP8G_ERR_ALIGNMENT;
    }
    if (N >= kMaxDim || (int64_t)E * N >= kMaxDim) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (K % 32 != 0) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(sfa, 16) || !aligned(sfb, 16) || !aligned(counts, 4)) return FP8G_ERR_ALIGNMENT;
    if (offsets_out != nullptr && !aligned(offsets_out, 4)) return FP8G_ERR_ALIGNMENT;
    if (tile_map_out != nullptr && !aligned(tile_map_out, 16)) return FP8G_ERR_ALIGNMENT;
    return FP8G_OK;
}

}  // namespace

// Kernel timing (fp8g_kernel_timing_begin / _end): events of the library
// recorded on the call's stream right before and right after the GEMM
// kernel's launch.
std::mutex g_timing_mu;
std::vector<cudaEvent_t> g_timing_start, g_timing_end;
int32_t g_timing_n = 0;
uint64_t g_timing_seq = 0;

template <class F>
cudaError_t timed_launch(cudaStream_t stream, F &&launch) {
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_timing_mu);
        if (g_timing_n > 0) {
            const int32_t i = (int32_t)(g_timing_seq++ % (uint64_t)g_timing_n);
            e0 = g_timing_start[i];
            e1 = g_timing_end[i];
        }
    }
    if (e0 != nullptr && cudaEventRecord(e0, stream) != cudaSuccess) return cudaGetLastError();
    const cudaError_t e = launch();
    if (e == cudaSuccess && e1 != nullptr) return cudaEventRecord(e1, stream);
    return e;
}

// Literal-scale GEMM through TF32: A' = TF32(dec(A) sfa), B' likewise (one
// HBM-bound pass each into a stream-ordered temporary from the library pool,
// fp32 words), then C = out(act(A' B'^T + bias)) on the pair kernel's TF32
// mode.  Each operand value is rounded once to TF32's 11 significant bits
// (relative error <= 2^-11), so every product is within 2^-10 of the exact
// one: inside the block-scaled tolerance 2^-8 sum |sa a| |sb b| + 1 ulp.
static fp8g_status run_tf32(const uint8_t *A, const uint8_t *B, const float *sfa, const float *sfb,
                     void *C, int out, int a_fmt, int b_fmt, const float *bias, int act,
                     int64_t M, int64_t N, int64_t K, const KernelChoice &kc, const DevInfo &di,
                     cudaStream_t stream) {
    cudaMemPool_t pool;
    fp8g_status st = scale_pool(di.dev, pool);
    if (st != FP8G_OK) return st;
    const size_t bytesA = ((size_t)M * (size_t)K * 4 + 255) / 256 * 256;
    const size_t bytesB = (size_t)N * (size_t)K * 4;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, bytesA + bytesB, pool, stream) != cudaSuccess)
        return FP8G_ERR_CUDA;
    float *tA = static_cast<float *>(ws);
    float *tB = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + bytesA);
    cudaError_t e = launch_dequant_tf32(A, sfa, M, K, a_fmt, tA, di.num_sms, stream);
    if (e == cudaSuccess) e = launch_dequant_tf32(B, sfb, N, K, b_fmt, tB, di.num_sms, stream);
    GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_kb = (int32_t)((K + 31) / 32);  // 32 fp32 values per 128-byte stage row
    p.npm = (int32_t)((M + kc.BM - 1) / kc.BM);
    p.npn = (int32_t)((N + kc.BN - 1) / kc.BN);
    p.T = (int64_t)p.npm * p.npn;
    p.split = 1;
    p.kb_per_split = p.num_kb;
    p.C = C;
    p.status = di.status;
    p.timeout_ns = timeout_ns();
    p.f4 = 3;
    p.bias = bias;
    p.act = act;
    p.c_rows = M;
    p.st32 = aligned(C, 32) && (N * (out == FP8G_OUT_F32 ? 4 : 2)) % 32 == 0;
    GemmMaps maps;
    if (e == cudaSuccess) {
        const uint64_t dA[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t dB[2] = {(uint64_t)K, (uint64_t)N};
        const uint32_t bA[2] = {32u, (uint32_t)kBM};
        const uint32_t bB[2] = {32u, (uint32_t)kc.b_rows};
        if (tmap_encode(tA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, 2, dA, bA,
                        CU_TENSOR_MAP_SWIZZLE_128B, di.dev, maps.A) != FP8G_OK ||
            tmap_encode(tB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, 2, dB, bB,
                        CU_TENSOR_MAP_SWIZZLE_128B, di.dev, maps.B) != FP8G_OK)
            e = cudaErrorInvalidValue;
        maps.SA = maps.A;
        maps.SB = maps.A;
    }
    if (e == cudaSuccess)
        e = timed_launch(stream, [&] {
            return launch_gemm(kModeTensor, out == FP8G_OUT_F32, maps, p, kc, stream);
        });
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return (e == cudaSuccess && ef == cudaSuccess) ? FP8G_OK : FP8G_ERR_CUDA;
}

fp8g_status run_gemm(int mode, const void *A, const void *B, const float *sa, const float *sb,
                     void *C, int out, int64_t M, int64_t N, int64_t K, const int32_t *counts,
                     int32_t E, int32_t *offsets_out, int32_t *tile_map_out, cudaStream_t stream,
                     void *scratch, size_t scratch_bytes, int a_fmt, int b_fmt,
                     const float *bias, int act, const int32_t *c_row_of, int64_t c_rows,
                     const FusedQuant *fq) {
    if (!valid_fmt(a_fmt) || !valid_fmt(b_fmt))
        return FP8G_ERR_INVALID_ARG;
    if (act != FP8G_ACT_NONE && act != FP8G_ACT_RELU && act != FP8G_ACT_GELU)
        return FP8G_ERR_INVALID_ARG;
    if (bias != nullptr && !aligned(bias, 4)) return FP8G_ERR_ALIGNMENT;
    fp8g_status st = check_packed(M > 0 ? A : B, B, M > 0 ? a_fmt : b_fmt, b_fmt, K);
    if (st != FP8G_OK) return st;
    DevInfo di;
    st = device_info(di);
    if (st != FP8G_OK) return st;
    KernelChoice kc = choose_kernel(mode, M, N, K, di.num_sms);
    if (fq != nullptr) kc.inl = false;  // the fused quantiser takes B's packed scale chunks
    // MXFP4 on CTA pairs runs at the FP4 rate (kind::mxf4, 256 K elements per
    // stage); every other E2M1 case takes the FP8-rate MMA with 4-bit loads
    const bool f4 = kc.pair && mode != kModeTensor && a_fmt == FP8G_E2M1 &&
                    b_fmt == FP8G_E2M1 && K % 256 == 0;
    GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_kb = f4 ? (int32_t)(K / 256) : (int32_t)((K + kBK - 1) / kBK);
    p.f4 = f4;
    const int32_t num_kg = f4 ? 2 * p.num_kb : p.num_kb;  // 128-wide K groups of the scales
    p.npm = (int32_t)((M + kc.BM - 1) / kc.BM);
    p.npn = (int32_t)((N + kc.BN - 1) / kc.BN);
    p.T = (int64_t)p.npm * p.npn;
    p.split = kc.split;
    p.kb_per_split = (p.num_kb + kc.split - 1) / kc.split;
    p.sa = sa;
    p.sb = sb;
    p.sfc = K / 32;
    p.C = C;
    p.counts = counts;
    p.E = E;
    p.offsets_out = offsets_out;
    p.tile_map_out = tile_map_out;
    p.status = di.status;
    p.timeout_ns = timeout_ns();
    p.ab_fmt = (mma_type(a_fmt) << 7) | (mma_type(b_fmt) << 10);
    p.a_gap8 = gap8(a_fmt);
    p.b_gap8 = gap8(b_fmt);
    p.bias = bias;
    p.act = act;
    p.c_row_of = c_row_of;
    p.c_rows = c_rows;
    p.st32 = aligned(C, 32) && (N * (out == FP8G_OUT_F32 ? 4 : 2)) % 32 == 0;
    if (fq != nullptr) {
        // the kernel quantises A itself (single CTAs only)
        if (mode != kModeGrouped || kc.pair || kc.split > 1 || f4) return FP8G_ERR_INVALID_ARG;
        p.xq = fq->x;
        p.xq_bf16 = fq->bf16;
        p.xq_rows = fq->rows;
        p.xq_src_rows = fq->src_rows;
        p.qa_out = fq->qa_out;
        p.sfa_out = fq->sfa_out;
    }

    GemmMaps maps;
    // grouped with zero rows, or A quantised in the kernel: A is never read
    // (a one-row map over B stands in)
    const bool a_read = M > 0 && fq == nullptr;
    const int64_t rows_a = a_read ? M : 1;
    const void *a_ptr = a_read ? A : B;
    const int a_map_fmt = a_read ? a_fmt : b_fmt;
    // operand maps count elements; the FP4-rate kernel views its packed
    // operands as dense bytes (K / 2 per row, 128 bytes = 256 codes per box row)
    const uint64_t kdim = f4 ? (uint64_t)(K / 2) : (uint64_t)K;
    const int map_fmt_a = f4 ? FP8G_E4M3 : a_map_fmt;
    const int map_fmt_b = f4 ? FP8G_E4M3 : b_fmt;
    {
        const uint64_t dA[2] = {kdim, (uint64_t)rows_a};
        const uint32_t bA[2] = {(uint32_t)kBK, (uint32_t)kBM};
        if ((st = tmap_operand(a_ptr, map_fmt_a, 2, dA, bA, di.dev, maps.A)) != FP8G_OK) return st;
    }
    if (mode == kModeGrouped) {
        const uint64_t dB[3] = {kdim, (uint64_t)N, (uint64_t)E};
        const uint32_t bB[3] = {(uint32_t)kBK, (uint32_t)kc.b_rows, 1u};
        if ((st = tmap_operand(B, map_fmt_b, 3, dB, bB, di.dev, maps.B)) != FP8G_OK) return st;
    } else {
        const uint64_t dB[2] = {kdim, (uint64_t)N};
        const uint32_t bB[2] = {(uint32_t)kBK, (uint32_t)kc.b_rows};
        if ((st = tmap_operand(B, map_fmt_b, 2, dB, bB, di.dev, maps.B)) != FP8G_OK) return st;
    }
    maps.SA = maps.A;
    maps.SB = maps.A;
    if (mode == kModeTensor) {
        const cudaError_t e = timed_launch(stream, [&] {
            return launch_gemm(mode, out == FP8G_OUT_F32, maps, p, kc, stream);
        });
        return e == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
    }
    if (kc.split > 1 || kc.inl) {
        // split-K or single CTAs on few tiles with short K: the GEMM converts
        // its own scale chunks from the fp32 scales (p.sa, p.sb; row stride p.sfc)
        const cudaError_t e = timed_launch(stream, [&] {
            return launch_gemm(mode, out == FP8G_OUT_F32, maps, p, kc, stream);
        });
        return e == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
    }
    // Block modes: pack the fp32 scales into UE8M0 chunks (a stream-ordered
    // temporary from the library pool), run the GEMM, return the temporary.
    const int32_t zB = mode == kModeGrouped ? E : 1;
    p.n_rtA = (int32_t)(mode == kModeGrouped ? M / kBM + E : (M + kBM - 1) / kBM);
    p.n_rtB = (int32_t)(((N + kc.BN - 1) / kc.BN) * (kc.BN / kBM));
    if (p.n_rtA > 65535 || p.n_rtB > 65535) return FP8G_ERR_UNSUPPORTED_SHAPE;
    // (the fused quantiser writes A's chunks into each stage itself)
    const size_t bytesA = fq != nullptr ? 0 : packed_scale_bytes(num_kg, p.n_rtA, 1);
    // single-CTA 256-wide tiles take B's scales replicated for one 128x256b
    // tensor-memory copy (4 KB per 256 rows and K step instead of 1 KB); CTA
    // pairs take plain 512-byte chunks (three warpx4 copies per K step)
    const bool repB = kc.BN == 256 && !kc.pair;
    const size_t bytesB = packed_scale_bytes(num_kg, p.n_rtB, zB) * (repB ? 4 : 1);
    void *ws = nullptr;
    if (scratch != nullptr) {
        // caller-provided scratch (the allocation-free entry point)
        if (bytesA + bytesB > scratch_bytes) return FP8G_ERR_UNSUPPORTED_SHAPE;
        ws = scratch;
    } else {
        cudaMemPool_t pool;
        if ((st = scale_pool(di.dev, pool)) != FP8G_OK) return st;
        if (cudaMallocFromPoolAsync(&ws, bytesA + bytesB, pool, stream) != cudaSuccess)
            return FP8G_ERR_CUDA;
    }
    uint8_t *pkA = static_cast<uint8_t *>(ws);
    uint8_t *pkB = pkA + bytesA;
    PackArgs pa{sa, M, 0, p.n_rtA, a_read ? 1 : 0, pkA, mode == kModeGrouped ? counts : nullptr, 0};
    PackArgs pb{sb, N, N, p.n_rtB, zB, pkB, nullptr, repB ? 1 : 0,
                mode == kModeGrouped ? counts : nullptr};
    cudaError_t e = launch_pack_scales(pa, pb, p.sfc, num_kg, E, di.status, stream);
    p.sfa_pk = pkA;
    p.sfb_pk = pkB;
    if (e == cudaSuccess && kc.pair) {
        // CTA pairs fetch the packed chunks by TMA: each array as rows of 128
        // uint32 (one 512-byte chunk per row)
        const uint64_t dSA[2] = {128u, (uint64_t)num_kg * (uint64_t)p.n_rtA};
        const uint32_t bSA[2] = {128u, 1u};
        const uint64_t dSB[2] = {128u, (uint64_t)zB * num_kg * (uint64_t)p.n_rtB};
        const uint32_t bSB[2] = {128u, 2u};  // 1 KB: the two 128-row chunks of a 256-row tile
        if (tmap_encode(pkA, CU_TENSOR_MAP_DATA_TYPE_UINT32, 32, 2, dSA, bSA,
                        CU_TENSOR_MAP_SWIZZLE_NONE, di.dev, maps.SA) != FP8G_OK ||
            tmap_encode(pkB, CU_TENSOR_MAP_DATA_TYPE_UINT32, 32, 2, dSB, bSB,
                        CU_TENSOR_MAP_SWIZZLE_NONE, di.dev, maps.SB) != FP8G_OK)
            e = cudaErrorInvalidValue;
    }
    if (e == cudaSuccess)
        e = timed_launch(stream, [&] { return launch_gemm(mode, out == FP8G_OUT_F32, maps, p, kc, stream); });
    const cudaError_t ef = scratch != nullptr ? cudaSuccess : cudaFreeAsync(ws, stream);
    return (e == cudaSuccess && ef == cudaSuccess) ? FP8G_OK : FP8G_ERR_CUDA;
}

// NVFP4 on CTA pairs (kind::mxf4nvf4 is issued with cta_group::2) whatever
// the shape: pack the E4M3 scale codes into the pair kernel's chunks (a
// stream-ordered temporary from the library pool), run the GEMM, return the
// temporary.  Grouped: A's row tiles are expert-local and B holds E matrices.
fp8g_status run_nvfp4(int mode, const void *A, const void *B, const uint8_t *sfa,
                      const uint8_t *sfb, const float *ga, const float *gb, void *C, int out,
                      const float *bias, int32_t act, int64_t M, int64_t N, int64_t K,
                      const int32_t *counts, int32_t E, int32_t *offsets_out,
                      int32_t *tile_map_out, cudaStream_t stream) {
    DevInfo di;
    fp8g_status st = device_info(di);
    if (st != FP8G_OK) return st;
    const bool grouped = mode == kModeGrouped;
    KernelChoice kc;
    kc.BM = 256;
    kc.BN = 256;
    kc.b_rows = 128;
    kc.split = 1;
    kc.cluster = 2;
    kc.pair = true;
    kc.inl = false;
    GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_kb = (int32_t)(K / 256);
    p.npm = (int32_t)((M + 255) / 256);
    p.npn = (int32_t)((N + 255) / 256);
    p.T = (int64_t)p.npm * p.npn;
    // grouped: at most M / 256 + E row tiles of 256 (the kernel counts them)
    const int64_t pairs = grouped ? (M / 256 + E) * p.npn : p.T;
    kc.grid = (int)(2 * (pairs < di.num_sms / 2 ? pairs : di.num_sms / 2));
    p.split = 1;
    p.kb_per_split = p.num_kb;
    p.C = C;
    p.counts = counts;
    p.E = E;
    p.offsets_out = offsets_out;
    p.tile_map_out = tile_map_out;
    p.c_rows = M;
    p.status = di.status;
    p.timeout_ns = timeout_ns();
    p.f4 = 2;
    p.ga = ga;
    p.gb = gb;
    p.bias = bias;
    p.act = act;
    p.st32 = aligned(C, 32) && (N * (out == FP8G_OUT_F32 ? 4 : 2)) % 32 == 0;
    const int32_t n_kg = (int32_t)(K / 64);  // 64-wide K groups: one MMA's four scales
    const int32_t zB = grouped ? E : 1;
    p.n_rtA = (int32_t)(grouped ? M / kBM + E : (M + kBM - 1) / kBM);
    p.n_rtB = (int32_t)(p.npn * 2);
    if (p.n_rtA > 65535 || p.n_rtB > 65535) return FP8G_ERR_UNSUPPORTED_SHAPE;
    // chunk rows are int32 TMA coordinates
    if ((int64_t)n_kg * p.n_rtA * 4 >= kMaxDim || (int64_t)zB * n_kg * p.n_rtB * 4 >= kMaxDim)
        return FP8G_ERR_UNSUPPORTED_SHAPE;
    GemmMaps maps;
    {
        // packed codes as dense bytes, K / 2 per row (128 bytes = 256 codes per
        // box row); grouped with zero rows: A is never read (B stands in)
        const uint64_t dA[2] = {(uint64_t)(K / 2), (uint64_t)(M > 0 ? M : 1)};
        const uint32_t bA[2] = {(uint32_t)kBK, (uint32_t)kBM};
        if ((st = tmap_operand(M > 0 ? A : B, FP8G_E4M3, 2, dA, bA, di.dev, maps.A)) != FP8G_OK)
            return st;
        if (grouped) {
            const uint64_t dB[3] = {(uint64_t)(K / 2), (uint64_t)N, (uint64_t)E};
            const uint32_t bB[3] = {(uint32_t)kBK, (uint32_t)kc.b_rows, 1u};
            if ((st = tmap_operand(B, FP8G_E4M3, 3, dB, bB, di.dev, maps.B)) != FP8G_OK) return st;
        } else {
            const uint64_t dB[2] = {(uint64_t)(K / 2), (uint64_t)N};
            const uint32_t bB[2] = {(uint32_t)kBK, (uint32_t)kc.b_rows};
            if ((st = tmap_operand(B, FP8G_E4M3, 2, dB, bB, di.dev, maps.B)) != FP8G_OK) return st;
        }
    }
    const size_t bytesA = packed_scale_bytes(n_kg, p.n_rtA, 1);
    const size_t bytesB = packed_scale_bytes(n_kg, p.n_rtB, zB);
    cudaMemPool_t pool;
    if ((st = scale_pool(di.dev, pool)) != FP8G_OK) return st;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, bytesA + bytesB, pool, stream) != cudaSuccess)
        return FP8G_ERR_CUDA;
    uint8_t *pkA = static_cast<uint8_t *>(ws);
    uint8_t *pkB = pkA + bytesA;
    cudaError_t e = launch_pack_nvfp4(sfa, M, p.n_rtA, pkA, grouped ? counts : nullptr, sfb, N,
                                      p.n_rtB, zB, pkB, n_kg, K / 16, E, stream);
    if (e == cudaSuccess) {
        // a stage's four K-group chunks are adjacent rows per 128-row tile
        const uint64_t dSA[2] = {128u, (uint64_t)n_kg * (uint64_t)p.n_rtA};
        const uint32_t bSA[2] = {128u, 4u};
        const uint64_t dSB[2] = {128u, (uint64_t)zB * n_kg * (uint64_t)p.n_rtB};
        const uint32_t bSB[2] = {128u, 8u};
        if (tmap_encode(pkA, CU_TENSOR_MAP_DATA_TYPE_UINT32, 32, 2, dSA, bSA,
                        CU_TENSOR_MAP_SWIZZLE_NONE, di.dev, maps.SA) != FP8G_OK ||
            tmap_encode(pkB, CU_TENSOR_MAP_DATA_TYPE_UINT32, 32, 2, dSB, bSB,
                        CU_TENSOR_MAP_SWIZZLE_NONE, di.dev, maps.SB) != FP8G_OK)
            e = cudaErrorInvalidValue;
    }
    if (e == cudaSuccess)
        e = timed_launch(stream, [&] {
            return launch_gemm(mode, out == FP8G_OUT_F32, maps, p, kc, stream);
        });
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return (e == cudaSuccess && ef == cudaSuccess) ? FP8G_OK : FP8G_ERR_CUDA;
}

fp8g_status check_blockscaled_args(const void *A, const void *B, const float *sfa,
                                  const float *sfb, const void *C, int out, int64_t M, int64_t N,
                                  int64_t K) {
    const fp8g_status st = check_common(A, B, C, out, M, N, K);
    if (st != FP8G_OK) return st;
    if (sfa == nullptr || sfb == nullptr) return FP8G_ERR_INVALID_ARG;
    if (K % 32 != 0) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(sfa, 16) || !aligned(sfb, 16)) return FP8G_ERR_ALIGNMENT;
    return FP8G_OK;
}

fp8g_status device_ready() {
    DevInfo di;
    return device_info(di);
}

}  // namespace fp8g

using namespace fp8g;

extern "C" {

fp8g_status fp8_gemm_ex(const void *A, const void *B, const float *scale_a,
                        const float *scale_b, void *C, int out, int32_t a_fmt, int32_t b_fmt,
                        const float *bias, int32_t act, int64_t M, int64_t N, int64_t K,
                        cudaStream_t stream) {
    fp8g_status st = check_common(A, B, C, out, M, N, K);
    if (st != FP8G_OK) return st;
    if (scale_a == nullptr || scale_b == nullptr) return FP8G_ERR_INVALID_ARG;
    if (!aligned(scale_a, 4) || !aligned(scale_b, 4)) return FP8G_ERR_ALIGNMENT;
    return run_gemm(kModeTensor, A, B, scale_a, scale_b, C, out, M, N, K, nullptr, 0, nullptr,
                    nullptr, stream, nullptr, 0, a_fmt, b_fmt, bias, act);
}

fp8g_status fp8_gemm_fmt(const void *A, const void *B, const float *scale_a,
                         const float *scale_b, void *C, int out, int32_t a_fmt, int32_t b_fmt,
                         int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return fp8_gemm_ex(A, B, scale_a, scale_b, C, out, a_fmt, b_fmt, nullptr, FP8G_ACT_NONE, M, N,
                       K, stream);
}

fp8g_status fp8_gemm(const void *A, const void *B, const float *scale_a, const float *scale_b,
                     void *C, int out, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return fp8_gemm_fmt(A, B, scale_a, scale_b, C, out, FP8G_E4M3, FP8G_E4M3, M, N, K, stream);
}

fp8g_status fp8_gemm_blockscaled_ex(const void *A, const void *B, const float *sfa,
                                    const float *sfb, void *C, int out, int32_t a_fmt,
                                    int32_t b_fmt, const float *bias, int32_t act, int64_t M,
                                    int64_t N, int64_t K, cudaStream_t stream) {
    const fp8g_status st = check_blockscaled_args(A, B, sfa, sfb, C, out, M, N, K);
    if (st != FP8G_OK) return st;
    return run_gemm(kModeBlock, A, B, sfa, sfb, C, out, M, N, K, nullptr, 0, nullptr, nullptr,
                    stream, nullptr, 0, a_fmt, b_fmt, bias, act);
}

fp8g_status fp8_gemm_blockscaled_promote(const void *A, const void *B, const float *sfa,
                                         const float *sfb, void *C, int out, int32_t a_fmt,
                                         int32_t b_fmt, const float *bias, int32_t act, int64_t M,
                                         int64_t N, int64_t K, cudaStream_t stream) {
    fp8g_status st = check_common(A, B, C, out, M, N, K);
    if (st != FP8G_OK) return st;
    if (sfa == nullptr || sfb == nullptr) return FP8G_ERR_INVALID_ARG;
    if (!valid_fmt(a_fmt) || !valid_fmt(b_fmt))
        return FP8G_ERR_INVALID_ARG;
    if (act != FP8G_ACT_NONE && act != FP8G_ACT_RELU && act != FP8G_ACT_GELU)
        return FP8G_ERR_INVALID_ARG;
    // the scales' rows (K/32 fp32) are TMA rows: 16-byte multiples
    if (K % 128 != 0) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if ((st = check_packed(A, B, a_fmt, b_fmt, K)) != FP8G_OK) return st;
    if (!aligned(sfa, 16) || !aligned(sfb, 16)) return FP8G_ERR_ALIGNMENT;
    if (bias != nullptr && !aligned(bias, 4)) return FP8G_ERR_ALIGNMENT;
    DevInfo di;
    if ((st = device_info(di)) != FP8G_OK) return st;
    // At least a wave of 256 x 256 tiles with 1-byte codes: fold each scale
    // into its operand once (dequantise to TF32) and run the TF32 tensor-core
    // GEMM on CTA pairs, instead of promoting every K block's partial on CUDA
    // cores (two fp32 operations per output per 32-wide K block)
    const KernelChoice kc = choose_kernel(kModeTensor, M, N, K, di.num_sms);
    if (kc.pair && (a_fmt == FP8G_E4M3 || a_fmt == FP8G_E5M2) &&
        (b_fmt == FP8G_E4M3 || b_fmt == FP8G_E5M2))
        return run_tf32(static_cast<const uint8_t *>(A), static_cast<const uint8_t *>(B), sfa, sfb,
                        C, out, a_fmt, b_fmt, bias, act, M, N, K, kc, di, stream);
    GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_kb = (int32_t)(K / kBK);
    p.npm = (int32_t)((M + kBM - 1) / kBM);
    p.npn = (int32_t)((N + 127) / 128);
    p.T = (int64_t)p.npm * p.npn;
    p.split = 1;
    p.sa = sfa;
    p.sb = sfb;
    p.sfc = K / 32;
    p.C = C;
    p.status = di.status;
    p.timeout_ns = timeout_ns();
    p.ab_fmt = (mma_type(a_fmt) << 7) | (mma_type(b_fmt) << 10);
    p.a_gap8 = gap8(a_fmt);
    p.b_gap8 = gap8(b_fmt);
    p.bias = bias;
    p.act = act;
    GemmMaps maps;
    const uint64_t dA[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t dB[2] = {(uint64_t)K, (uint64_t)N};
    const uint32_t box[2] = {(uint32_t)kBK, 128u};
    const uint64_t dSA[2] = {(uint64_t)(K / 32), (uint64_t)M};
    const uint64_t dSB[2] = {(uint64_t)(K / 32), (uint64_t)N};
    const uint32_t bS[2] = {4u, 128u};  // 4 K blocks x 128 rows of fp32
    if ((st = tmap_operand(A, a_fmt, 2, dA, box, di.dev, maps.A)) != FP8G_OK) return st;
    if ((st = tmap_operand(B, b_fmt, 2, dB, box, di.dev, maps.B)) != FP8G_OK) return st;
    if ((st = tmap_encode(sfa, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, 2, dSA, bS,
                          CU_TENSOR_MAP_SWIZZLE_NONE, di.dev, maps.SA)) != FP8G_OK)
        return st;
    if ((st = tmap_encode(sfb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, 2, dSB, bS,
                          CU_TENSOR_MAP_SWIZZLE_NONE, di.dev, maps.SB)) != FP8G_OK)
        return st;
    const int grid = (int)(p.T < di.num_sms ? p.T : di.num_sms);
    const cudaError_t e = timed_launch(
        stream, [&] { return launch_gemm_promote(out == FP8G_OUT_F32, maps, p, grid, stream); });
    return e == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

fp8g_status fp8_gemm_nvfp4(const void *A, const void *B, const uint8_t *sfa, const uint8_t *sfb,
                           const float *ga, const float *gb, void *C, int out, const float *bias,
                           int32_t act, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    fp8g_status st = check_common(A, B, C, out, M, N, K);
    if (st != FP8G_OK) return st;
    if (sfa == nullptr || sfb == nullptr || ga == nullptr || gb == nullptr)
        return FP8G_ERR_INVALID_ARG;
    if (act != FP8G_ACT_NONE && act != FP8G_ACT_RELU && act != FP8G_ACT_GELU)
        return FP8G_ERR_INVALID_ARG;
    if (K % 256 != 0) return FP8G_ERR_UNSUPPORTED_SHAPE;
    // scale rows are read 16 bytes at a time (K / 16 bytes per row, K % 256 == 0)
    if (!aligned(A, 32) || !aligned(B, 32) || !aligned(sfa, 16) || !aligned(sfb, 16) ||
        !aligned(ga, 4) || !aligned(gb, 4))
        return FP8G_ERR_ALIGNMENT;
    if (bias != nullptr && !aligned(bias, 4)) return FP8G_ERR_ALIGNMENT;
    return run_nvfp4(kModeBlock, A, B, sfa, sfb, ga, gb, C, out, bias, act, M, N, K, nullptr, 1,
                     nullptr, nullptr, stream);
}

fp8g_status fp8_grouped_gemm_nvfp4(const void *A, const void *B, const uint8_t *sfa,
                                   const uint8_t *sfb, const float *ga, const float *gb, void *C,
                                   int out, const float *bias, int32_t act, const int32_t *counts,
                                   int32_t E, int64_t N, int64_t K, int64_t total_rows,
                                   int32_t *offsets_out, int32_t *tile_map_out,
                                   cudaStream_t stream) {
    if (counts == nullptr || sfa == nullptr || sfb == nullptr || ga == nullptr || gb == nullptr)
        return FP8G_ERR_INVALID_ARG;
    if (E < 1) return FP8G_ERR_INVALID_ARG;
    if (E > FP8G_MAX_EXPERTS) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (total_rows < 0) return FP8G_ERR_INVALID_ARG;
    if (act != FP8G_ACT_NONE && act != FP8G_ACT_RELU && act != FP8G_ACT_GELU)
        return FP8G_ERR_INVALID_ARG;
    if (total_rows > 0) {
        fp8g_status st = check_common(A, B, C, out, total_rows, N, K);
        if (st != FP8G_OK) return st;
        if (!aligned(A, 32)) return FP8G_ERR_ALIGNMENT;
    } else {
        if (B == nullptr) return FP8G_ERR_INVALID_ARG;
        if (out != FP8G_OUT_BF16 && out != FP8G_OUT_F32) return FP8G_ERR_INVALID_ARG;
        if (N < 1 || K < 1) return FP8G_ERR_INVALID_ARG;
    }
    if (N >= kMaxDim || K >= kMaxDim || (int64_t)E * N >= kMaxDim) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (K % 256 != 0) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(B, 32) || !aligned(sfa, 16) || !aligned(sfb, 16) || !aligned(ga, 4) ||
        !aligned(gb, 4) || !aligned(counts, 4))
        return FP8G_ERR_ALIGNMENT;
    if (bias != nullptr && !aligned(bias, 4)) return FP8G_ERR_ALIGNMENT;
    if (offsets_out != nullptr && !aligned(offsets_out, 4)) return FP8G_ERR_ALIGNMENT;
    if (tile_map_out != nullptr && !aligned(tile_map_out, 16)) return FP8G_ERR_ALIGNMENT;
    return run_nvfp4(kModeGrouped, A, B, sfa, sfb, ga, gb, C, out, bias, act, total_rows, N, K,
                     counts, E, offsets_out, tile_map_out, stream);
}

fp8g_status fp8g_quantize_nvfp4(const void *x, int32_t in_dtype, int64_t rows, int64_t cols,
                                uint8_t *q, uint8_t *sf, float *g, cudaStream_t stream) {
    if (x == nullptr || q == nullptr || sf == nullptr || g == nullptr) return FP8G_ERR_INVALID_ARG;
    if (in_dtype != FP8G_IN_F32 && in_dtype != FP8G_IN_BF16) return FP8G_ERR_INVALID_ARG;
    if (rows < 1 || cols < 1) return FP8G_ERR_INVALID_ARG;
    if (cols % 16 != 0) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (rows >= ((int64_t)1 << 40) / cols || rows > INT32_MAX) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || !aligned(q, 4) || !aligned(g, 4)) return FP8G_ERR_ALIGNMENT;
    DevInfo di;
    fp8g_status st = device_info(di);
    if (st != FP8G_OK) return st;
    const cudaError_t e = launch_quantize_nvfp4(x, in_dtype == FP8G_IN_BF16, rows, cols, q, sf, g,
                                                di.status, di.num_sms, stream);
    return e == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

fp8g_status fp8_gemm_blockscaled_fmt(const void *A, const void *B, const float *sfa,
                                     const float *sfb, void *C, int out, int32_t a_fmt,
                                     int32_t b_fmt, int64_t M, int64_t N, int64_t K,
                                     cudaStream_t stream) {
    return fp8_gemm_blockscaled_ex(A, B, sfa, sfb, C, out, a_fmt, b_fmt, nullptr, FP8G_ACT_NONE,
                                   M, N, K, stream);
}

fp8g_status fp8_gemm_blockscaled(const void *A, const void *B, const float *sfa,
                                 const float *sfb, void *C, int out, int64_t M, int64_t N,
                                 int64_t K, cudaStream_t stream) {
    return fp8_gemm_blockscaled_fmt(A, B, sfa, sfb, C, out, FP8G_E4M3, FP8G_E4M3, M, N, K,
                                    stream);
}

fp8g_status fp8_grouped_gemm(const void *A, const void *B, const float *sfa, const float *sfb,
                             void *C, int out, const int32_t *counts, int32_t E, int64_t N,
                             int64_t K, int64_t total_rows, int32_t *offsets_out,
                             int32_t *tile_map_out, cudaStream_t stream) {
    return fp8_grouped_gemm_fmt(A, B, sfa, sfb, C, out, FP8G_E4M3, FP8G_E4M3, counts, E, N, K,
                                total_rows, offsets_out, tile_map_out, stream);
}

fp8g_status fp8_grouped_gemm_fmt(const void *A, const void *B, const float *sfa,
                                 const float *sfb, void *C, int out, int32_t a_fmt, int32_t b_fmt,
                                 const int32_t *counts, int32_t E, int64_t N, int64_t K,
                                 int64_t total_rows, int32_t *offsets_out, int32_t *tile_map_out,
                                 cudaStream_t stream) {
    return fp8_grouped_gemm_ex(A, B, sfa, sfb, C, out, a_fmt, b_fmt, nullptr, FP8G_ACT_NONE,
                               counts, E, N, K, total_rows, offsets_out, tile_map_out, stream);
}

fp8g_status fp8_grouped_gemm_ex(const void *A, const void *B, const float *sfa,
                                const float *sfb, void *C, int out, int32_t a_fmt, int32_t b_fmt,
                                const float *bias, int32_t act, const int32_t *counts, int32_t E,
                                int64_t N, int64_t K, int64_t total_rows, int32_t *offsets_out,
                                int32_t *tile_map_out, cudaStream_t stream) {
    return fp8_grouped_gemm_scatter(A, B, sfa, sfb, C, out, a_fmt, b_fmt, bias, act, counts, E, N,
                                    K, total_rows, nullptr, total_rows, offsets_out, tile_map_out,
                                    stream);
}

fp8g_status fp8_grouped_gemm_scatter(const void *A, const void *B, const float *sfa,
                                     const float *sfb, void *C, int out, int32_t a_fmt,
                                     int32_t b_fmt, const float *bias, int32_t act,
                                     const int32_t *counts, int32_t E, int64_t N, int64_t K,
                                     int64_t total_rows, const int32_t *c_row_of, int64_t c_rows,
                                     int32_t *offsets_out, int32_t *tile_map_out,
                                     cudaStream_t stream) {
    const fp8g_status st = check_grouped_args(A, B, sfa, sfb, C, out, counts, E, N, K, total_rows,
                                              c_row_of, c_rows, offsets_out, tile_map_out);
    if (st != FP8G_OK) return st;
    return run_gemm(kModeGrouped, A, B, sfa, sfb, C, out, total_rows, N, K, counts, E,
                    offsets_out, tile_map_out, stream, nullptr, 0, a_fmt, b_fmt, bias, act,
                    c_row_of, c_row_of != nullptr ? c_rows : total_rows);
}

fp8g_status fp8_grouped_gemm_quant(const void *X, int32_t x_dtype, int64_t x_rows,
                                   const int32_t *rows, const void *B, const float *sfb, void *C,
                                   int out, int32_t b_fmt, const float *bias, int32_t act,
                                   const int32_t *counts, int32_t E, int64_t N, int64_t K,
                                   int64_t total_rows, const int32_t *c_row_of, int64_t c_rows,
                                   uint8_t *qa_out, float *sfa_out, int32_t *offsets_out,
                                   int32_t *tile_map_out, int32_t flags, cudaStream_t stream) {
    if (x_dtype != FP8G_IN_F32 && x_dtype != FP8G_IN_BF16) return FP8G_ERR_INVALID_ARG;
    if (flags != 0 && flags != FP8G_QUANT_FUSED) return FP8G_ERR_INVALID_ARG;
    if ((qa_out == nullptr) != (sfa_out == nullptr)) return FP8G_ERR_INVALID_ARG;
    if (total_rows > 0) {
        if (X == nullptr || x_rows < 1) return FP8G_ERR_INVALID_ARG;
        if (rows == nullptr && total_rows > x_rows) return FP8G_ERR_INVALID_ARG;
        if (x_rows >= kMaxDim) return FP8G_ERR_UNSUPPORTED_SHAPE;
        if (!aligned(X, 16)) return FP8G_ERR_ALIGNMENT;
        if (rows != nullptr && !aligned(rows, 4)) return FP8G_ERR_ALIGNMENT;
    }
    if (qa_out != nullptr && (!aligned(qa_out, 16) || !aligned(sfa_out, 16)))
        return FP8G_ERR_ALIGNMENT;
    // the grouped GEMM's own rules; the quantised A (X's place when it stays
    // in shared memory) stands in for A and its scales
    const void *a_arg = qa_out != nullptr ? static_cast<const void *>(qa_out) : X;
    const float *sfa_arg = sfa_out != nullptr ? sfa_out : sfb;
    fp8g_status st = check_grouped_args(a_arg, B, sfa_arg, sfb, C, out, counts, E, N, K,
                                        total_rows, c_row_of, c_rows, offsets_out, tile_map_out);
    if (st != FP8G_OK) return st;
    // the rest of the GEMM's host rules, before anything is launched
    if (!valid_fmt(b_fmt)) return FP8G_ERR_INVALID_ARG;
    if (act != FP8G_ACT_NONE && act != FP8G_ACT_RELU && act != FP8G_ACT_GELU)
        return FP8G_ERR_INVALID_ARG;
    if (bias != nullptr && !aligned(bias, 4)) return FP8G_ERR_ALIGNMENT;
    if ((st = check_packed(B, B, FP8G_E4M3, b_fmt, K)) != FP8G_OK) return st;
    if (total_rows / kBM + E > 65535) return FP8G_ERR_UNSUPPORTED_SHAPE;
    const int64_t c_rows_eff = c_row_of != nullptr ? c_rows : total_rows;
    DevInfo di;
    if ((st = device_info(di)) != FP8G_OK) return st;
    const KernelChoice kc = choose_kernel(kModeGrouped, total_rows, N, K, di.num_sms);
    if (flags == FP8G_QUANT_FUSED && total_rows > 0 && !kc.pair) {
        // one kernel: the GEMM quantises each tile of A it multiplies
        const FusedQuant fq{X, x_dtype == FP8G_IN_BF16 ? 1 : 0, rows, x_rows, qa_out, sfa_out};
        return run_gemm(kModeGrouped, nullptr, B, nullptr, sfb, C, out, total_rows, N, K, counts,
                        E, offsets_out, tile_map_out, stream, nullptr, 0, FP8G_E4M3, b_fmt, bias,
                        act, c_row_of, c_rows_eff, &fq);
    }
    // two kernels: gather-quantise, then the grouped GEMM
    uint8_t *qa = qa_out;
    float *sa = sfa_out;
    void *tmp = nullptr;
    if (total_rows > 0 && qa == nullptr) {
        cudaMemPool_t pool;
        if ((st = scale_pool(di.dev, pool)) != FP8G_OK) return st;
        const size_t code_bytes = ((size_t)total_rows * (size_t)K + 255) / 256 * 256;
        const size_t scale_bytes = (size_t)total_rows * (size_t)(K / 32) * 4;
        if (cudaMallocFromPoolAsync(&tmp, code_bytes + scale_bytes, pool, stream) != cudaSuccess)
            return FP8G_ERR_CUDA;
        qa = static_cast<uint8_t *>(tmp);
        sa = reinterpret_cast<float *>(qa + code_bytes);
    }
    if (total_rows > 0)
        st = fp8g_quantize_rows(X, x_dtype, x_rows, K, rows, total_rows, 32, FP8G_E4M3, qa, sa,
                                stream);
    if (st == FP8G_OK)
        st = run_gemm(kModeGrouped, qa, B, total_rows > 0 ? sa : sfb, sfb, C, out, total_rows, N,
                      K, counts, E, offsets_out, tile_map_out, stream, nullptr, 0, FP8G_E4M3,
                      b_fmt, bias, act, c_row_of, c_rows_eff);
    if (tmp != nullptr && cudaFreeAsync(tmp, stream) != cudaSuccess && st == FP8G_OK)
        st = FP8G_ERR_CUDA;
    return st;
}



fp8g_status fp8g_grouped_plan(int64_t N, int64_t K, int64_t total_rows, int32_t E, int32_t *BM,
                              int32_t *BN, int32_t *G, int64_t *max_tiles) {
    if (N < 1 || K < 1 || total_rows < 0 || E < 1) return FP8G_ERR_INVALID_ARG;
    if (E > FP8G_MAX_EXPERTS) return FP8G_ERR_UNSUPPORTED_SHAPE;
    DevInfo di;
    const int sms = device_info(di) == FP8G_OK ? di.num_sms : 148;
    const KernelChoice kc = choose_kernel(kModeGrouped, total_rows, N, K, sms);
    if (BM) *BM = kc.BM;
    if (BN) *BN = kc.BN;
    if (G) *G = kRasterG;
    // sum_e ceil(M_e / BM) <= floor(total_rows / BM) + E
    if (max_tiles) *max_tiles = (total_rows / kc.BM + E) * ((N + kc.BN - 1) / kc.BN);
    return FP8G_OK;
}

fp8g_status fp8g_gemm_plan(int block, int64_t M, int64_t N, int64_t K, int32_t *BM, int32_t *BN,
                           int32_t *G, int32_t *split_k, int32_t *grid) {
    if (M < 1 || N < 1 || K < 1 || (block != 0 && block != 1)) return FP8G_ERR_INVALID_ARG;
    DevInfo di;
    fp8g_status st = device_info(di);
    if (st != FP8G_OK) return st;
    const KernelChoice kc = choose_kernel(block ? kModeBlock : kModeTensor, M, N, K, di.num_sms);
    if (BM) *BM = kc.BM;
    if (BN) *BN = kc.BN;
    if (G) *G = kRasterG;
    if (split_k) *split_k = kc.split;
    if (grid) *grid = kc.grid;
    return FP8G_OK;
}

fp8g_status fp8g_quantize_e4m3(const float *x, int64_t rows, int64_t cols, int32_t block,
                               uint8_t *q, float *scales, cudaStream_t stream) {
    return fp8g_quantize(x, rows, cols, block, FP8G_E4M3, q, scales, stream);
}

fp8g_status fp8g_quantize(const float *x, int64_t rows, int64_t cols, int32_t block, int32_t fmt,
                          uint8_t *q, float *scales, cudaStream_t stream) {
    return fp8g_quantize_rows(x, FP8G_IN_F32, rows, cols, nullptr, rows, block, fmt, q, scales,
                              stream);
}

fp8g_status fp8g_quantize_rows(const void *x, int32_t in_dtype, int64_t x_rows, int64_t cols,
                               const int32_t *rows, int64_t n_rows, int32_t block, int32_t fmt,
                               uint8_t *q, float *scales, cudaStream_t stream) {
    if (x == nullptr || q == nullptr || scales == nullptr) return FP8G_ERR_INVALID_ARG;
    if (!valid_fmt(fmt)) return FP8G_ERR_INVALID_ARG;
    if (in_dtype != FP8G_IN_F32 && in_dtype != FP8G_IN_BF16) return FP8G_ERR_INVALID_ARG;
    if (x_rows < 1 || n_rows < 1 || cols < 1) return FP8G_ERR_INVALID_ARG;
    if (rows == nullptr && n_rows > x_rows) return FP8G_ERR_INVALID_ARG;
    if (rows != nullptr && !aligned(rows, 4)) return FP8G_ERR_ALIGNMENT;
    if (block != 0 && block != 32 && block != FP8G_BLOCK32_LITERAL) return FP8G_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q, 8) || !aligned(scales, 4)) return FP8G_ERR_ALIGNMENT;
    if (block != 0 && cols % 32 != 0) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (cols % 8 != 0) return FP8G_ERR_UNSUPPORTED_SHAPE;
    if (x_rows >= ((int64_t)1 << 40) / cols || n_rows >= ((int64_t)1 << 40) / cols ||
        x_rows > INT32_MAX)
        return FP8G_ERR_UNSUPPORTED_SHAPE;
    DevInfo di;
    fp8g_status st = device_info(di);
    if (st != FP8G_OK) return st;
    const cudaError_t e = launch_quantize_rows(x, in_dtype == FP8G_IN_BF16, x_rows, cols, rows,
                                               n_rows, block, fmt, q, scales, di.status,
                                               di.num_sms, stream);
    return e == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

fp8g_status fp8_gemm_status(cudaStream_t stream, int32_t *detail) {
    DevInfo di;
    fp8g_status st = device_info(di);
    if (st != FP8G_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8G_ERR_CUDA;
    unsigned int w[2] = {0u, 0u};
    if (cudaMemcpy(w, di.status, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess)
        return FP8G_ERR_CUDA;
    if (w[0] != 0u) {
        const unsigned int zero[2] = {0u, 0u};
        if (cudaMemcpy(di.status, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return FP8G_ERR_CUDA;
    }
    if (detail) *detail = (int32_t)w[1];
    return (fp8g_status)w[0];
}

const char *fp8g_status_string(fp8g_status s) {
    switch (s) {
        case FP8G_OK: return "ok";
        case FP8G_ERR_INVALID_ARG: return "invalid argument";
        case FP8G_ERR_ALIGNMENT: return "alignment rule broken (16-byte pointers and row strides)";
        case FP8G_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case FP8G_ERR_SCALE_FORMAT: return "block scale is not a positive power of two";
        case FP8G_ERR_CUDA: return "CUDA call failed";
        case FP8G_ERR_TIMEOUT: return "device-side wait timed out; kernel aborted";
        case FP8G_ERR_DEVICE: return "no usable sm_103 device";
    }
    return "unknown status";
}

fp8g_status fp8g_kernel_timing_begin(int32_t n) {
    if (n < 1 || n > (1 << 20)) return FP8G_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_timing_mu);
    if (g_timing_n != 0) return FP8G_ERR_INVALID_ARG;  // already on
    g_timing_start.assign((size_t)n, nullptr);
    g_timing_end.assign((size_t)n, nullptr);
    for (int32_t i = 0; i < n; ++i)
        if (cudaEventCreate(&g_timing_start[i]) != cudaSuccess ||
            cudaEventCreate(&g_timing_end[i]) != cudaSuccess) {
            for (auto e : g_timing_start)
                if (e) cudaEventDestroy(e);
            for (auto e : g_timing_end)
                if (e) cudaEventDestroy(e);
            g_timing_start.clear();
            g_timing_end.clear();
            return FP8G_ERR_CUDA;
        }
    g_timing_n = n;
    g_timing_seq = 0;
    return FP8G_OK;
}

fp8g_status fp8g_kernel_timing_end(float *ms, int32_t cap, int32_t *count) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    if (g_timing_n == 0) return FP8G_ERR_INVALID_ARG;
    const int32_t rec = (int32_t)(g_timing_seq < (uint64_t)g_timing_n ? g_timing_seq : g_timing_n);
    fp8g_status st = FP8G_OK;
    int32_t got = 0;
    for (int32_t i = 0; i < rec && i < cap && ms != nullptr; ++i) {
        float t = 0.0f;
        if (cudaEventSynchronize(g_timing_end[i]) != cudaSuccess ||
            cudaEventElapsedTime(&t, g_timing_start[i], g_timing_end[i]) != cudaSuccess) {
            st = FP8G_ERR_CUDA;
            break;
        }
        ms[got++] = t;
    }
    if (count) *count = got;
    for (auto e : g_timing_start) cudaEventDestroy(e);
    for (auto e : g_timing_end) cudaEventDestroy(e);
    g_timing_start.clear();
    g_timing_end.clear();
    g_timing_n = 0;
    g_timing_seq = 0;
    return st;
}

fp8g_status fp8g_wait_selftest(uint32_t timeout_us, cudaStream_t stream) {
    if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return FP8G_ERR_INVALID_ARG;
    DevInfo di;
    const fp8g_status st = device_info(di);
    if (st != FP8G_OK) return st;
    const cudaError_t e = launch_wait_selftest(di.status, (uint64_t)timeout_us * 1000ull, stream);
    return e == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

void fp8g_set_wait_timeout_ms(uint32_t ms) {
    if (ms == 0) {
        g_timeout_ns.store(0, std::memory_order_relaxed);
        (void)timeout_ns();
    } else {
        g_timeout_ns.store((uint64_t)ms * 1000000ull, std::memory_order_relaxed);
    }
}

void fp8g_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_cache.clear();
    for (int d = 0; d < kMaxDevices; ++d)
        if (g_pool_ok[d]) cudaMemPoolTrimTo(g_pool[d], 0);
}

int fp8g_version(void) { return 100; }

}  // extern "C"
