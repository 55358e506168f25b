// launch.h - the kernels' host-side entry (defined in kernels.cu).
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

#include "plan.h"

namespace mcc1d {

// Enqueues the main and reduce kernels of plan `p` on `stream`. Pointers have
// been validated by the caller. Returns kOk or kErrCuda.
int32_t launch_bwd(const Plan &p, const void *gradY, const void *x, const void *weight,
                   const uint8_t *mask, void *gradX, void *gradWeight, void *workspace,
                   cudaStream_t stream);

}  // namespace mcc1d
