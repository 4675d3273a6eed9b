// selftest.cu -- a check of the bounded-wait protocol itself: a kernel that
// waits on an mbarrier phase nothing will complete, with the same sleeping
// bounded wait the library's kernels use, but a limit the caller chooses,
// and reports the expiry into the device error word as they do.  Nothing is
// copied, so nothing is left in flight when it returns.
#include "common.cuh"
#include "kernels.h"
#include "w4q.h"

namespace w4q {

namespace {

__global__ void wait_expiry_kernel(unsigned *err, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);  // one expected arrival, which never comes
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_sleep(b, 0u, limit_ns))
        report_error(err, ERR_FULL_WAIT);
}

}  // namespace

}  // namespace w4q

extern "C" int w4q_selftest_wait_expiry(unsigned limit_us, void *stream)
{
    if (limit_us == 0 || limit_us > 100000)
        return W4Q_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return W4Q_ERR_CUDA;
    unsigned *err = w4q::device_error_word(dev);
    if (err == nullptr)
        return W4Q_ERR_CUDA;
    w4q::wait_expiry_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        err, 1000ull * limit_us);
    return cudaGetLastError() == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}
