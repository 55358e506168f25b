// device.cpp - current_context_id() (through the runtime's driver entry-point
// query: the library does not link the driver library directly) and the
// device check of the SM count the plans assume.
#include "device.h"

#include <cuda_runtime_api.h>

#include <atomic>
#include <mutex>

#include "plan.h"

namespace mcc1d {

unsigned long long current_context_id()
{
    typedef int (*CtxGetCurrentFn)(void **);
    typedef int (*CtxGetIdFn)(void *, unsigned long long *);
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
        (void)cudaGetLastError();
    });
    if (!get_current || !get_id)
        return 0;
    void *ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != 0 || ctx == nullptr || get_id(ctx, &id) != 0)
        return 0;
    return id;
}

int32_t check_sm_count(int32_t sm_count)
{
    return sm_count >= kNumSMs ? kOk : kErrDevice;
}

int32_t current_device_sm_count()
{
    static std::atomic<int32_t> cache[64];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev < 64) {
        const int32_t v = cache[dev].load(std::memory_order_acquire);
        if (v > 0)
            return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev < 64)
        cache[dev].store(n, std::memory_order_release);
    return n;
}

int32_t check_current_device()
{
    const int32_t n = current_device_sm_count();
    return n > 0 ? check_sm_count(n) : kErrCuda;
}

}  // namespace mcc1d
