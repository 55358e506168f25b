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

#include "device.h"
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

// The array's device address, cached per device together with the unique id
// of the context it was looked up in. A device reset (cudaDeviceReset, or a
// host framework that releases and re-creates the primary context) loads the
// library's module again in a new context, where the array may sit at a new
// address; the changed context id makes the next call look it up again.
struct ScratchSlot {
    unsigned long long ctx_id;   // 0: unknown
    void *addr;
};
ScratchSlot g_scratch[kMaxDevices];

// Device address of g_noalloc_scratch on the current device. The first call
// on a device (and the first after its context was re-created) looks it up
// with that device current; later calls reuse it.
int32_t scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return kErrCuda;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchSlot &slot = g_scratch[dev];
    if (slot.addr == nullptr || ctx == 0 || slot.ctx_id != ctx) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return kErrCuda;
        slot.addr = ptr;
        // the lookup makes the device's primary context current if none was
        slot.ctx_id = ctx != 0 ? ctx : current_context_id();
    }
    *out = slot.addr;
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
    const int32_t dv = check_current_device();
    if (dv != kOk)
        return dv;
    void *scratch = nullptr;
    const int32_t sa = scratch_address(&scratch);
    if (sa != kOk)
        return sa;
    // Nothing in the scratch has to start at zero: each call writes every
    // status word and partial it later reads.
    return launch_bwd(p, dense_layout(S, B, H), gradY, x, weight, mask_or_null, gradX, gradWeight,
                      scratch, static_cast<cudaStream_t>(stream));
}
