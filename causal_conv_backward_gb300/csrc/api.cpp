// api.cpp - the extern "C" entry points declared in include/mcc1d.h.
//
// Both phases validate in the order null pointers, dtype, shape, alignment,
// workspace; nothing touches a device before every check has passed.
#include <cuda_runtime_api.h>
#include <stdint.h>

#include "launch.h"
#include "mcc1d.h"
#include "plan.h"

using namespace mcc1d;

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

extern "C" int32_t mcc1d_bwd_workspace_size(int64_t S, int64_t B, int64_t H, int64_t W,
                                            int32_t dtype, int32_t has_mask, uint64_t *bytes_out)
{
    (void)has_mask;
    if (!bytes_out)
        return kErrNull;
    Plan p;
    const int32_t st = make_plan(S, B, H, W, dtype, &p);
    if (st != kOk)
        return st;
    *bytes_out = p.ws_bytes;
    return kOk;
}

extern "C" int32_t mcc1d_bwd(const void *gradY, const void *x, const void *weight,
                             const uint8_t *mask_or_null, void *gradX, void *gradWeight,
                             void *workspace, void *stream, int64_t S, int64_t B, int64_t H,
                             int64_t W, int32_t dtype, uint64_t workspace_bytes)
{
    if (!gradY || !x || !weight || !gradX || !gradWeight || !workspace)
        return kErrNull;
    Plan p;
    const int32_t st = make_plan(S, B, H, W, dtype, &p);
    if (st != kOk)
        return st;
    if (!aligned16(gradY) || !aligned16(x) || !aligned16(weight) || !aligned16(gradX) ||
        !aligned16(gradWeight) || !aligned16(workspace))
        return kErrInvalid;
    if (workspace_bytes < p.ws_bytes)
        return kErrWorkspace;
    return launch_bwd(p, gradY, x, weight, mask_or_null, gradX, gradWeight, workspace,
                      static_cast<cudaStream_t>(stream));
}

extern "C" int32_t mcc1d_bwd_device_status(const void *workspace, void *stream, int32_t *status_out)
{
    if (!workspace || !status_out)
        return kErrNull;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return kErrCuda;
    int32_t v = 0;
    if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return kErrCuda;
    *status_out = v;
    return kOk;
}

extern "C" const char *mcc1d_status_string(int32_t status)
{
    switch (status) {
    case kOk: return "MCC1D_OK";
    case kErrNull: return "MCC1D_ERR_PARAM_NULLPTR: a required pointer is null";
    case kErrInvalid: return "MCC1D_ERR_PARAM_INVALID: unsupported dtype or a pointer not 16-byte aligned";
    case kErrShape: return "MCC1D_ERR_INNER_TILING_ERROR: shape outside B 1..32, B*S 1..524288, H 384..24576 (H%64==0), W==3";
    case kErrWorkspace: return "MCC1D_ERR_WORKSPACE: workspace smaller than mcc1d_bwd_workspace_size reported";
    case kErrCuda: return "MCC1D_ERR_CUDA: a CUDA runtime call failed";
    case kErrTimeout: return "MCC1D_ERR_DEVICE_TIMEOUT: a device-side wait gave up; outputs are not valid";
    default: return "unknown mcc1d status";
    }
}

extern "C" int32_t mcc1d_version(void) { return 100; }
