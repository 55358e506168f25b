// selftest.cu - a self-test of the bounded device-side wait that every kernel
// of the library relies on: one thread waits on a shared-memory mbarrier with
// the same helper (mbar_wait_bounded) the main, forward and direct kernels
// use. With `arrive` set the thread arrives first and the wait succeeds; with
// it clear nothing ever arrives, the wait gives up after kWaitLimitNs and the
// kernel reports kErrTimeout through its status word and returns, leaving the
// context usable. No asynchronous copy or other thread is involved.
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "launch.h"
#include "plan.h"

namespace mcc1d {

__global__ void __launch_bounds__(32) mcc1d_wait_selftest(int32_t *status, int32_t arrive)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0)
        return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (arrive)
        mbar_arrive(b);
    const bool ok = mbar_wait_bounded(b, 0);
    *status = ok ? kOk : kErrTimeout;
}

int32_t launch_wait_selftest(int32_t *status, int32_t arrive, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    cfg.stream = stream;
    if (cudaLaunchKernelEx(&cfg, mcc1d_wait_selftest, status, arrive) != cudaSuccess)
        return kErrCuda;
    return kOk;
}

}  // namespace mcc1d
