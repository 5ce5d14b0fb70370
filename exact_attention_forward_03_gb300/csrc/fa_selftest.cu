// fa_selftest.cu -- a kernel whose only job is to let a bounded wait run out, so
// that the timeout path (status bit, host error code, a context that stays
// usable) can be tested without faulting or hanging the GPU.
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

// One warp: lane 0 initialises an mbarrier that expects one arrival, and no one
// ever arrives.  Every lane waits for its first phase with the time limit given,
// then records the timeout the way the attention kernels do.
__global__ void __launch_bounds__(32) fa_selftest_timeout_kernel(int *status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar_storage;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    const unsigned long long t0 = globaltimer_ns();
    bool done = false;
    for (uint32_t n = 1; !done; ++n) {
        if (mbar_try_wait(bar, 0)) break;
        if ((n & 15u) == 0 && globaltimer_ns() - t0 > limit_ns) done = true;
    }
    if (done && threadIdx.x == 0) atomicOr(status, kDevErrTimeout);
}

cudaError_t launch_selftest_timeout(int *status, int limit_ms, cudaStream_t stream) {
    return launch_kernel(fa_selftest_timeout_kernel, dim3(1), dim3(32), 0, stream, status,
                         (unsigned long long)limit_ms * 1000000ull);
}

}  // namespace fa
