// misc.cu -- status strings, device query, and the bounded-wait check used
// by the fault-handling tests.
#include "common.cuh"

namespace moe {

// One thread initialises an mbarrier that expects one arrival which never
// comes, then waits on it with the same bounded wait the pipelined kernels
// use.  On expiry the status bit is set and the kernel returns normally.
__global__ void bounded_wait_kernel(int64_t timeout_ns, int32_t *dev_status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait_bounded(&bar, 0, (uint64_t)timeout_ns)) dev_flag(dev_status, MOE_DEV_TIMEOUT);
    }
}

} // namespace moe

using namespace moe;

MOE_API const char *moe_status_str(moe_status s)
{
    switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "null pointer";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_ALIGN: return "misaligned pointer or leading dimension";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA launch or driver error";
    case MOE_ERR_UNSUPPORTED: return "unsupported option";
    default: return "unknown status";
    }
}

MOE_API moe_status moe_debug_bounded_wait(int64_t timeout_ns, int32_t *dev_status, void *stream)
{
    if (!dev_status) return MOE_ERR_NULL;
    if (timeout_ns < 0 || timeout_ns > 10LL * 1000 * 1000 * 1000) return MOE_ERR_SHAPE;
    bounded_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(timeout_ns, dev_status);
    return launch_status();
}

MOE_API int moe_device_sm_count(void) { return sm_count(); }
