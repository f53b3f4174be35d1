// Allocation-free variant of the block-scaled GEMM.
//
// fp8_gemm_blockscaled repacks the caller's fp32 scales into the tensor
// core's UE8M0 layout in a temporary taken from a device memory pool.  Some
// callers cannot have the library allocate device memory at all: for example
// code running under a strict memory budget or a custom allocator that owns
// every device byte, or an embedding that forbids allocation calls on its hot
// path.  fp8_gemm_blockscaled_noalloc does the same work but keeps the packed
// scales in the fixed device array below, which is part of the library image:
// it exists on every GPU that loads the library, from load until process exit,
// and no call allocates or frees anything.
#include <mutex>

#include "internal.h"

namespace fp8g {
namespace {

// Packed-scale scratch: at most (ceil(M/128) + 8 ceil(N/256)) * ceil(K/128)
// * 512 bytes must fit (16 MiB; M = N = K = 8192 needs 10 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDev] = {};

// Device address of the scratch array on the current device.  The array's
// name is only a host-side stand-in in host code; its device address comes
// from cudaGetSymbolAddress, once per device, with that device current.
fp8g_status noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return FP8G_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return FP8G_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FP8G_OK;
}

}  // namespace
}  // namespace fp8g

using namespace fp8g;

extern "C" {

fp8g_status fp8_gemm_blockscaled_noalloc(const void *A, const void *B, const float *sfa,
                                         const float *sfb, void *C, int out, int64_t M, int64_t N,
                                         int64_t K, cudaStream_t stream) {
    // the checks of fp8_gemm_blockscaled, in its order, then the device's
    fp8g_status st = check_blockscaled_args(A, B, sfa, sfb, C, out, M, N, K);
    if (st != FP8G_OK) return st;
    if ((st = device_ready()) != FP8G_OK) return st;
    void *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != FP8G_OK) return st;
    // run_gemm returns FP8G_ERR_UNSUPPORTED_SHAPE, before launching anything,
    // when the packed scales would not fit in the array.
    return run_gemm(kModeBlock, A, B, sfa, sfb, C, out, M, N, K, nullptr, 0, nullptr, nullptr,
                    stream, scratch, kNoAllocScratchBytes);
}

}  // extern "C"
