// launch.h - the kernels' host-side entry (defined in kernels.cu).
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

#include "plan.h"

namespace mcc1d {

// Enqueues the main and reduce kernels of plan `p` on `stream`. gradY and x
// must be row-streamable under `L` (unit H stride, 16-byte aligned rows);
// weight and mask may have any strides. Pointers have been validated by the
// caller. Returns kOk or kErrCuda.
int32_t launch_bwd(const Plan &p, const Layout &L, const void *gradY, const void *x,
                   const void *weight, const uint8_t *mask, void *gradX, void *gradWeight,
                   void *workspace, cudaStream_t stream);

// Enqueues the reduce kernel of plan `p` (programmatic dependent launch after
// the main kernel on `stream`): sums the partials in `workspace` and writes
// gradWeight (any device-accessible address). Returns kOk or kErrCuda.
int32_t launch_reduce(const Plan &p, void *workspace, void *gradWeight, cudaStream_t stream);

// Enqueues the backward on dense tensors that may live in page-locked host
// memory (read and written in place by the kernel), then the reduce. Pointers
// are device-accessible addresses. Returns kOk or kErrCuda.
int32_t launch_direct(const Plan &p, const void *gradY, const void *x, const void *weight,
                      const uint8_t *mask, void *gradX, void *gradWeight, void *workspace,
                      cudaStream_t stream);

// Enqueues a gather of a strided 16-bit [S,B,H] tensor into a dense one
// (dst 16-byte aligned). Returns kOk or kErrCuda.
int32_t launch_pack(const void *src, const int64_t strides[3], void *dst, int64_t S, int64_t B,
                    int64_t H, cudaStream_t stream);

// The forward's shared-memory ring for plan `p` (its own rows per stage and
// depth; the backward's ring fields of the plan do not apply to it).
struct FwdRing {
    int32_t rows_per_stage, stages;
    uint32_t slot_bytes, off_halo, off_mask, off_bar, smem_bytes;
};
FwdRing fwd_ring(const Plan &p);
// Shared memory of the forward's smallest ring (two slots) for plan `p`.
uint32_t fwd_ring_min_bytes(const Plan &p);
// Whether the forward stores y rows with bulk copies out of its ring (wide
// rows) rather than with per-thread stores.
bool fwd_bulk_store(const Plan &p);
// The forward kernel's form for plan `p`: plain, bulk y stores (wide rows at
// W = 3), or deep stages (W >= 6 on H-blocks of kFwdDeepMinHbWidth channels
// and more).
enum { kFwdPlain = 0, kFwdBulkStores = 1, kFwdDeep = 2 };
int fwd_variant(const Plan &p);
// One thread waiting on an mbarrier with the library's bounded wait; writes
// kOk (arrive != 0: it arrives first) or kErrTimeout (nothing arrives) to the
// device word `status`.
int32_t launch_wait_selftest(int32_t *status, int32_t arrive, cudaStream_t stream);
// Registers per thread of the forward kernel instance for (dtype, vec, W,
// fwd_variant), from the runtime (0 when unknown).
int fwd_kernel_regs(int dtype, int vec, int W, int variant);
// Enqueues the forward kernel of plan `p`; the inputs are read with layout L
// (x with unit H stride and 16-byte aligned rows), y is dense. `status` is a
// device word the kernel ORs kErrTimeout into if a wait gives up, or null.
int32_t launch_fwd(const Plan &p, const Layout &L, const void *x, const void *weight, const uint8_t *mask,
                   void *y, int32_t *status, cudaStream_t stream);

}  // namespace mcc1d
