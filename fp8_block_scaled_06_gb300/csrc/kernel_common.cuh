// Device helpers shared by the GEMM kernels: the grouped raster order of
// output tiles and the bounded mbarrier waits with their error reporting.
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace fp8g {

// Grouped raster order: bands of G tile-rows; inside a band walk down one
// tile-column, then move to the next column.  (Tile counts fit in 31 bits.)
__device__ __forceinline__ void raster(int32_t t, int32_t npm, int32_t npn, int32_t G, int32_t &pm,
                                       int32_t &pn) {
    const int32_t band = G * npn;
    const int32_t grp = t / band;
    const int32_t first = grp * G;
    const int32_t height = min(npm - first, G);
    const int32_t in_band = t - grp * band;
    pm = first + in_band % height;
    pn = in_band / height;
}

__device__ __forceinline__ void record_error(const GemmParams &p, unsigned code, unsigned detail) {
    if (atomicCAS(&p.status[0], 0u, code) == 0u) atomicExch(&p.status[1], detail);
}

// Bounded wait on an mbarrier phase.  Returns false when this CTA is aborting
// (another role timed out) or when this wait itself exceeded the limit.
// sleep_ns > 0 backs off between polls (for roles that wait a whole tile).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         const GemmParams &p, unsigned detail,
                                         uint32_t sleep_ns = 0) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            record_error(p, FP8G_ERR_TIMEOUT, detail);
            return false;
        }
        if (sleep_ns) __nanosleep(sleep_ns);
    }
}

// Warp-uniform bounded wait: lane 0 waits, the outcome is broadcast, and the
// warp re-converges before any .sync.aligned tcgen05 instruction follows.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              volatile int *abort_flag, const GemmParams &p,
                                              unsigned detail, uint32_t sleep_ns = 0) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort_flag, p, detail, sleep_ns) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

}  // namespace fp8g
