// noalloc.cu - mcc1d_bwd_noalloc: the backward without a caller workspace.
//
// Some callers cannot allocate device memory when they call the backward:
// code that runs inside a runtime or framework that owns every device
// allocation, or a caller whose memory budget is fixed to the tensors it is
// handed. They cannot provide the workspace mcc1d_bwd asks for. This entry
// point gives them the same kernels with their scratch (per-CTA gradWeight
// partial sums and status words) in a fixed array of device memory that is
// part of this library's image, so the call itself allocates nothing.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "launch.h"
#include "mcc1d.h"
#include "plan.h"

using namespace mcc1d;

// The scratch: every GPU that loads the library holds these bytes until the
// process exits. Device code could name it directly; host code needs its
// device address, looked up once per device below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MCC1D_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device. The first call
// on a device looks it up with that device current; later calls reuse it.
int32_t scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return kErrCuda;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return kErrCuda;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return kOk;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
}  // namespace

extern "C" int32_t mcc1d_bwd_noalloc(const void *gradY, const void *x, const void *weight,
                                     const uint8_t *mask_or_null, void *gradX, void *gradWeight,
                                     void *stream, int64_t S, int64_t B, int64_t H, int64_t W,
                                     int32_t dtype)
{
    if (!gradY || !x || !weight || !gradX || !gradWeight)
        return kErrNull;
    Plan p;
    const int32_t st = make_plan(S, B, H, W, dtype, &p);
    if (st != kOk)
        return st;
    if (!aligned16(gradY) || !aligned16(x) || !aligned16(weight) || !aligned16(gradX) ||
        !aligned16(gradWeight))
        return kErrInvalid;
    // The shape's scratch must fit the fixed array.
    if (p.ws_bytes > (uint64_t)MCC1D_NOALLOC_SCRATCH_BYTES)
        return kErrWorkspace;
    void *scratch = nullptr;
    const int32_t sa = scratch_address(&scratch);
    if (sa != kOk)
        return sa;
    // Nothing in the scratch has to start at zero: each call writes every
    // status word and partial it later reads.
    return launch_bwd(p, dense_layout(S, B, H), gradY, x, weight, mask_or_null, gradX, gradWeight,
                      scratch, static_cast<cudaStream_t>(stream));
}
