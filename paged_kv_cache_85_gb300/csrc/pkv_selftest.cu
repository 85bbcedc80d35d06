// pkv_selftest_bounded_wait: runs the kernels' bounded mbarrier wait on a
// barrier that nothing completes (or, as a control, one that a lane has
// already arrived on), so a test can see the timeout path report
// PKV_FLAG_TIMEOUT and return.  No copy is in flight, no other warp or CTA
// is involved, and the wait's limit is capped at 0.1 s.
#include <cuda_runtime.h>

#include "pkv.h"
#include "pkv_ptx.cuh"
#include "pkv_selftest.h"

namespace pkv {
pkv_status report_error(pkv_status s, const char *msg);

__global__ void __launch_bounds__(32, 1)
    selftest_bounded_wait_kernel(uint64_t limit_ns, int arrive, int32_t *err_flag,
                                 uint64_t *waited_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncwarp();
    if (arrive && lane == 0)
        mbar_arrive(&bar);
    __syncwarp();
    const uint64_t t0 = global_timer_ns();
    // the same pattern as the pipeline warps: every lane waits, the warp agrees
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar, 0, limit_ns));
    const uint64_t t1 = global_timer_ns();
    if (lane == 0) {
        if (!ok)
            flag_error(err_flag, PKV_FLAG_TIMEOUT);
        if (waited_ns)
            *waited_ns = t1 - t0;
    }
}
} // namespace pkv

extern "C" pkv_status pkv_selftest_bounded_wait(uint64_t limit_ns, int arrive, int32_t *err_flag,
                                                uint64_t *waited_ns, void *stream)
{
    if (limit_ns < 1 || limit_ns > 100000000ull)
        return pkv::report_error(PKV_ERR_INVALID_ARG,
                                 "selftest_bounded_wait: limit_ns must be in [1, 1e8]");
    if (!err_flag || (reinterpret_cast<uintptr_t>(err_flag) & 3u) ||
        (reinterpret_cast<uintptr_t>(waited_ns) & 7u))
        return pkv::report_error(PKV_ERR_INVALID_ARG,
                                 "selftest_bounded_wait: err_flag is required; pointers aligned");
    pkv::selftest_bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        limit_ns, arrive, err_flag, waited_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return pkv::report_error(PKV_ERR_CUDA, cudaGetErrorString(e));
    return PKV_OK;
}
