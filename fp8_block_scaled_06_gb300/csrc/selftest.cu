// Self-test of the bounded-wait and status mechanism every GEMM kernel uses:
// one warp completes one mbarrier wait (an arrival it makes itself), then
// waits on a barrier that nothing arrives at.  That wait gives up after the
// requested limit and records FP8G_ERR_TIMEOUT (detail kSelftestDetail) in
// the device status word, exactly as a GEMM role would; the kernel then
// returns normally.  No fault, trap or unbounded wait is involved.
#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace fp8g {

namespace {

constexpr unsigned kSelftestDetail = 0xDEADu;

__global__ void __launch_bounds__(32) wait_selftest_kernel(GemmParams p) {
    __shared__ uint64_t bars[2];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&bars[0]), 1);
        ptx::mbar_init(ptx::smem_addr(&bars[1]), 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        ptx::mbar_arrive(ptx::smem_addr(&bars[0]));
        // completes: the arrival above finished phase 0
        if (!wait_bar(ptx::smem_addr(&bars[0]), 0, &abort_flag, p, 1u))
            record_error(p, FP8G_ERR_DEVICE, 1u);
        // never completes: runs out after p.timeout_ns and records the timeout
        wait_bar(ptx::smem_addr(&bars[1]), 0, &abort_flag, p, kSelftestDetail);
    }
    __syncwarp();
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned int *status, uint64_t timeout_ns, cudaStream_t s) {
    GemmParams p{};
    p.status = status;
    p.timeout_ns = timeout_ns;
    wait_selftest_kernel<<<1, 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace fp8g
