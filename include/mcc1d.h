/*
 * mcc1d.h - masked causal depthwise conv1d backward (and forward) for NVIDIA GB300.
 *
 * C ABI of libmcc1d.so. The operation is the one defined on the CANN operator
 * page "aclnnMaskedCausalConv1dBackward", section 功能说明 (function
 * description), 计算公式 (formulas). With gradY, x, gradX laid out [S,B,H],
 * weight [W,H] and the optional bool mask [B,S]:
 *
 *   gradYMasked(i,j,h) = mask(j,i) * gradY(i,j,h)
 *   gradX(i,j,h)       = sum over k = 0..W-1 of gradYMasked(i+k,j,h) * weight(W-1-k,h)
 *   gradWeight(k,h)    = sum over j < B, i < S of gradYMasked(i+W-1-k,j,h) * x(i,j,h)
 *
 * Terms whose S index falls outside [0,S) are zero; batches never mix; H is
 * the depthwise (elementwise) axis. W is 3 on the page-shaped calls, the only
 * width the page supports; the strided calls (mcc1d_bwd_ex, mcc1d_fwd_ex) and
 * the forward take any 1 <= W <= 8 with the same formulas.
 *
 * The page's two-phase call (函数原型 / function prototypes) maps to
 *   1. mcc1d_bwd_workspace_size: validate and size the workspace (host only);
 *   2. mcc1d_bwd: validate again and enqueue the computation on a stream.
 * Raw pointers carry no shapes, so the second phase takes the shape again in
 * place of the page's opaque executor object.
 *
 * Conventions shared by every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates no memory and keeps no state between calls.
 *  - Tensors are dense and row-major: gradY, x, gradX [S,B,H]; weight and
 *    gradWeight [W,H]; mask [B,S] with one byte per position, nonzero = keep
 *    (the _ex calls take strided inputs through a descriptor; their outputs
 *    stay dense).
 *  - gradY, x, weight, gradX, gradWeight and workspace must be 16-byte
 *    aligned; the mask may have any alignment.
 *  - The data type (bf16 or fp16) is the same for all five 16-bit tensors, as
 *    the page's parameter table (参数说明) requires. Accumulation is fp32;
 *    outputs are rounded to nearest even.
 *  - gradX and gradWeight must not overlap each other, an input or the
 *    workspace (not checked).
 *  - Results are deterministic: the same inputs, shape and device give
 *    bitwise-identical outputs (the page promises a deterministic
 *    implementation, 约束说明 / constraints). No floating-point atomics are
 *    used; every sum has a fixed order that depends on the shape only.
 *  - Status codes mirror the page's return codes (返回值 / return values);
 *    codes >= 561003 are this library's own.
 *
 * Shape limits (约束说明 / constraints): 1 <= B <= 32, 1 <= B*S <= 524288,
 * 384 <= H <= 24576 with H % 64 == 0, W == 3 (1 <= W <= 8 where stated
 * above). Anything else is
 * MCC1D_ERR_INNER_TILING_ERROR. The page also promises that inputs hold no
 * inf or NaN and that no intermediate value overflows the 16-bit type; the
 * library relies on that and does not check it.
 */
#ifndef MCC1D_H
#define MCC1D_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of gradY, x, weight, gradX and gradWeight (the page allows
 * BFLOAT16 and FLOAT16). */
typedef enum { MCC1D_BF16 = 0, MCC1D_FP16 = 1 } mcc1d_dtype;

typedef enum {
    MCC1D_OK = 0,
    /* A required pointer is null (page code ACLNN_ERR_PARAM_NULLPTR). */
    MCC1D_ERR_PARAM_NULLPTR = 161001,
    /* Unsupported dtype, or a tensor pointer that is not 16-byte aligned
     * (page code ACLNN_ERR_PARAM_INVALID: dtype or format out of range). */
    MCC1D_ERR_PARAM_INVALID = 161002,
    /* Shape outside the supported range (page code ACLNN_ERR_INNER_TILING_ERROR). */
    MCC1D_ERR_INNER_TILING_ERROR = 561002,
    /* The workspace passed to mcc1d_bwd is smaller than the size phase 1 reported. */
    MCC1D_ERR_WORKSPACE = 561003,
    /* A CUDA runtime call failed (launch, attribute or copy); nothing is
     * guaranteed about the outputs. */
    MCC1D_ERR_CUDA = 561100,
    /* Reported by mcc1d_bwd_device_status: a device-side wait of the last
     * call gave up after its time limit and the outputs are not valid. */
    MCC1D_ERR_DEVICE_TIMEOUT = 561101,
    /* The current device has fewer SMs than the launch plans are cut for
     * (MCC1D_PLAN_SMS): part of every grid would run as a second wave at
     * about twice the time. Returned by every call that launches, before
     * anything is enqueued. */
    MCC1D_ERR_DEVICE = 561102
} mcc1d_status;

/* SMs the launch plans assume (GB300: two dies of 76). The plans are a
 * function of the shape alone, so results never depend on the device. */
#define MCC1D_PLAN_SMS 152

/*
 * Phase 1 (page: aclnnMaskedCausalConv1dBackwardGetWorkspaceSize).
 *
 * Validates the shape and dtype and writes to *bytes_out the size of device
 * workspace that mcc1d_bwd needs for this shape. Runs on the host only and
 * touches no device. has_mask (0 or 1) is accepted to mirror the page's
 * optional mask; the size does not depend on it.
 *
 * Errors: MCC1D_ERR_PARAM_NULLPTR if bytes_out is null;
 * MCC1D_ERR_PARAM_INVALID for an unknown dtype; MCC1D_ERR_INNER_TILING_ERROR
 * for a shape outside the limits above. *bytes_out is untouched on error.
 */
int32_t mcc1d_bwd_workspace_size(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype,
                                 int32_t has_mask, uint64_t *bytes_out);

/*
 * Phase 2 (page: aclnnMaskedCausalConv1dBackward).
 *
 * Enqueues the backward on `stream` (a cudaStream_t; NULL is the legacy
 * default stream) of the current device and returns without waiting. All
 * tensor pointers must belong to the current device.
 *
 *   gradY        [S,B,H] input, dtype
 *   x            [S,B,H] input, dtype (the forward's input)
 *   weight       [W,H]   input, dtype
 *   mask_or_null [B,S]   input bytes, nonzero = keep; NULL keeps every position
 *   gradX        [S,B,H] output, dtype; every element is written
 *   gradWeight   [W,H]   output, dtype; every element is written
 *   workspace    device scratch of at least workspace_bytes bytes, where
 *                workspace_bytes >= the size phase 1 reported for this shape.
 *                Its contents on entry are ignored and are overwritten; it must
 *                not be used by anything else until the call has completed on
 *                the stream. Two calls that may run at the same time need two
 *                workspaces.
 *
 * Returns MCC1D_OK once the work is enqueued. Errors (nothing is enqueued):
 * MCC1D_ERR_PARAM_NULLPTR (a null tensor or workspace pointer),
 * MCC1D_ERR_PARAM_INVALID (dtype, or a pointer not 16-byte aligned),
 * MCC1D_ERR_INNER_TILING_ERROR (shape), MCC1D_ERR_WORKSPACE (workspace_bytes
 * too small), MCC1D_ERR_DEVICE (the current device has fewer than
 * MCC1D_PLAN_SMS SMs), MCC1D_ERR_CUDA (a launch failed; the CUDA error is
 * left for cudaGetLastError to report).
 */
int32_t mcc1d_bwd(const void *gradY, const void *x, const void *weight,
                  const uint8_t *mask_or_null, void *gradX, void *gradWeight,
                  void *workspace, void *stream,
                  int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype,
                  uint64_t workspace_bytes);

/*
 * The backward on tensors that may live in host memory (an extension of the
 * page's call, which takes device tensors). gradY, x, weight, mask, gradX and
 * gradWeight may each be page-locked host memory (cudaMallocHost,
 * cudaHostAlloc or cudaHostRegister) or device memory of the current device;
 * the kernel reads and writes them in place over the host link, so the
 * inputs stream in, gradX streams out and the arithmetic runs at the same
 * time, with no staging copies. The workspace is device memory, sized by
 * mcc1d_bwd_workspace_size. Arguments, layouts, results (within the same
 * tolerances; gradWeight may differ from mcc1d_bwd in its last bit, its
 * partial sums are grouped differently) and errors are those of mcc1d_bwd,
 * plus MCC1D_ERR_PARAM_INVALID for a pointer the device cannot access
 * (pageable host memory, or memory of another device). Host buffers must
 * stay valid and untouched until the call completes on `stream`.
 */
int32_t mcc1d_bwd_host(const void *gradY, const void *x, const void *weight,
                       const uint8_t *mask_or_null, void *gradX, void *gradWeight,
                       void *workspace, void *stream,
                       int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype,
                       uint64_t workspace_bytes);

/*
 * Tensors of one call with explicit strides: the page's inputs may be
 * non-contiguous (the 非连续Tensor column of its parameter table), its
 * outputs may not. Strides count ELEMENTS for the 16-bit tensors and BYTES for
 * the mask, outermost dimension first; no stride may be negative (a zero
 * stride repeats data). Strides of dimensions of size 1 are ignored.
 *
 *   gradY, x      [S,B,H] inputs: strides {S, B, H}
 *   weight        [W,H]   input:  strides {W, H}
 *   mask          [B,S]   input bytes or NULL: strides {B, S}
 *   gradX         [S,B,H] output, dense (strides {B*H, H, 1})
 *   gradWeight    [W,H]   output, dense (strides {H, 1})
 *
 * gradY and x with unit H stride and 16-byte aligned rows (base pointer and
 * the S and B strides in bytes multiples of 16, e.g. a [B,S,H] buffer seen
 * as [S,B,H], or an H-slice of a wider tensor) are streamed in place. Any
 * other layout of gradY or x is first gathered into a dense copy inside the
 * workspace, which then includes S*B*H*2 bytes per such tensor. weight and
 * mask are read in place with any strides.
 */
typedef struct mcc1d_tensors {
    const void *gradY;
    int64_t gradY_strides[3];
    const void *x;
    int64_t x_strides[3];
    const void *weight;
    int64_t weight_strides[2];
    const uint8_t *mask;
    int64_t mask_strides[2];
    void *gradX;
    void *gradWeight;
} mcc1d_tensors;

/*
 * Phase 1 for strided tensors (page: the same GetWorkspaceSize call, which
 * receives the tensors themselves). The workspace size depends on the
 * layouts and base pointers of gradY and x. Validation as
 * mcc1d_bwd_workspace_size except for the kernel width: the strided calls
 * take any 1 <= W <= 8 (the page supports W = 3 only today, 约束说明 /
 * constraints; its formulas, 计算公式, are written for any W: gradX sums W
 * taps and gradWeight has W rows). Plus: MCC1D_ERR_PARAM_NULLPTR for a null
 * descriptor or required pointer; MCC1D_ERR_PARAM_INVALID for a negative
 * stride, a 16-bit input pointer that is not 2-byte aligned, or an output
 * pointer that is not 16-byte aligned.
 */
int32_t mcc1d_bwd_ex_workspace_size(const mcc1d_tensors *t, int64_t S, int64_t B, int64_t H,
                                    int64_t W, int32_t dtype, uint64_t *bytes_out);

/*
 * Phase 2 for strided tensors: as mcc1d_bwd, with the tensors described by
 * `t`. Results are bitwise identical to mcc1d_bwd on dense copies of the same
 * values. Errors as mcc1d_bwd_ex_workspace_size and mcc1d_bwd.
 */
int32_t mcc1d_bwd_ex(const mcc1d_tensors *t, int64_t S, int64_t B, int64_t H, int64_t W,
                     int32_t dtype, void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * Device-side status of the last mcc1d_bwd that used `workspace`: waits for
 * `stream` to finish, then copies the status word that the call left in the
 * workspace to *status_out (MCC1D_OK, or MCC1D_ERR_DEVICE_TIMEOUT when a
 * bounded device-side wait gave up). Synchronous; meant for tests and
 * debugging. Returns MCC1D_ERR_PARAM_NULLPTR for null pointers and
 * MCC1D_ERR_CUDA if the copy or the synchronisation failed.
 */
int32_t mcc1d_bwd_device_status(const void *workspace, void *stream, int32_t *status_out);

/*
 * Backward without a workspace argument. The operator page has no
 * counterpart to this call: it is for callers that cannot allocate device
 * memory at call time (code running inside a runtime or framework that owns
 * every device allocation, or whose memory budget is fixed to the tensors it
 * is handed) and so cannot supply the workspace that mcc1d_bwd needs.
 *
 * Arguments and results are those of mcc1d_bwd without workspace and
 * workspace_bytes; the call allocates nothing. Its scratch (the per-CTA
 * gradWeight partial sums and status words) lives instead in one fixed
 * device array of MCC1D_NOALLOC_SCRATCH_BYTES (8 MiB) inside the library
 * image, which every GPU that loads the library holds until the process
 * exits.
 *
 *  - A shape whose mcc1d_bwd_workspace_size exceeds MCC1D_NOALLOC_SCRATCH_BYTES
 *    is rejected with MCC1D_ERR_WORKSPACE before anything is enqueued. Every
 *    shape within the limits above needs at most about 4.7 MB, so all of them
 *    fit; the check guards against a future plan needing more.
 *  - All calls on a device share the one array. Calls that may overlap on the
 *    GPU (different streams, or host threads with no ordering between them)
 *    race on it and give wrong results: order them on one stream or with
 *    events.
 *  - The array keeps what the last call left in it; the kernels write every
 *    scratch word before they read it, so nothing needs clearing between calls.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture begins. The address is cached with the id of
 *    the context it was found in: after a device reset (cudaDeviceReset, or
 *    a framework re-creating the primary context) the next call looks it up
 *    again, since the new context may place the array elsewhere.
 *  - A device-side wait that gives up (the bounded waits described under
 *    mcc1d_bwd_device_status) goes unreported on this call: the status words
 *    live in the shared array, which no caller can read, so the call returns
 *    MCC1D_OK with gradX and gradWeight incomplete. Callers that need to
 *    detect that use mcc1d_bwd and mcc1d_bwd_device_status.
 * Errors: as mcc1d_bwd, plus MCC1D_ERR_WORKSPACE for a shape too large for the
 * array and MCC1D_ERR_CUDA if the address lookup fails.
 */
#define MCC1D_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
int32_t mcc1d_bwd_noalloc(const void *gradY, const void *x, const void *weight,
                          const uint8_t *mask_or_null, void *gradX, void *gradWeight,
                          void *stream, int64_t S, int64_t B, int64_t H, int64_t W,
                          int32_t dtype);

/*
 * Forward of the same operator (MaskedCausalConv1d, the forward the page
 * names; its mask is the convolution's output mask): for every channel h,
 *
 *   y(t,j,h) = mask(j,t) * sum over k = 0..W-1 of weight(k,h) * x(t-W+1+k, j, h)
 *
 * with x zero before t = 0, a causal depthwise convolution with W-1 positions
 * of left padding. mcc1d_bwd computes exactly the gradients of this map. The
 * page prints no forward API; this one follows mcc1d_bwd's conventions:
 *
 *   x            [S,B,H] input, dtype, dense, 16-byte aligned
 *   weight       [W,H]   input, dtype, dense, 16-byte aligned
 *   mask_or_null [B,S]   input bytes, nonzero = keep; NULL keeps every position
 *   y            [S,B,H] output, dtype, dense, 16-byte aligned; every element written
 *   device_status_or_null  a device int32 the kernel sets to
 *                MCC1D_ERR_DEVICE_TIMEOUT if a bounded device-side wait gives
 *                up (it is never cleared: zero it before the call to use it), or NULL
 *
 * Enqueued on `stream`; no workspace; deterministic; y within 1 ulp of the
 * exact value rounded once. Errors and shape limits as mcc1d_bwd, except the
 * kernel width: any 1 <= W <= 8 (the page's W = 3, and the widths the strided
 * backward accepts, so a caller gets both directions of the same conv).
 */
int32_t mcc1d_fwd(const void *x, const void *weight, const uint8_t *mask_or_null, void *y,
                  void *stream, int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype,
                  int32_t *device_status_or_null);

/*
 * The forward on strided inputs, as mcc1d_bwd_ex is the backward's: strides
 * in elements (bytes for the mask), outermost first, negative strides
 * rejected, strides of size-1 dimensions ignored.
 *
 *   x       [S,B,H] input: strides {S, B, H}; 2-byte aligned
 *   weight  [W,H]   input: strides {W, H}; 2-byte aligned; read in place
 *   mask    [B,S]   input bytes or NULL: strides {B, S}; read in place
 *   y       [S,B,H] output, dense (strides {B*H, H, 1}), 16-byte aligned
 *
 * x with unit H stride and 16-byte aligned rows (base and the S and B
 * strides in bytes multiples of 16) is streamed in place and the call needs
 * no workspace (size 0; workspace may be NULL). Any other x is first gathered
 * into a dense copy in the workspace: S*B*H*2 bytes rounded up to 256. y is
 * bitwise identical to mcc1d_fwd's on a dense copy of the same values.
 */
typedef struct mcc1d_fwd_tensors {
    const void *x;
    int64_t x_strides[3];
    const void *weight;
    int64_t weight_strides[2];
    const uint8_t *mask;
    int64_t mask_strides[2];
    void *y;
} mcc1d_fwd_tensors;

/* Workspace bytes of mcc1d_fwd_ex for these tensors (0 when x streams in
 * place). Validation as mcc1d_fwd (1 <= W <= 8) plus the stride and
 * alignment rules above. Host only. */
int32_t mcc1d_fwd_ex_workspace_size(const mcc1d_fwd_tensors *t, int64_t S, int64_t B, int64_t H,
                                    int64_t W, int32_t dtype, uint64_t *bytes_out);

/* Enqueue the forward on the tensors described by `t` (see above); errors as
 * mcc1d_fwd_ex_workspace_size and mcc1d_fwd, MCC1D_ERR_WORKSPACE if a needed
 * workspace is smaller than mcc1d_fwd_ex_workspace_size. */
int32_t mcc1d_fwd_ex(const mcc1d_fwd_tensors *t, int64_t S, int64_t B, int64_t H, int64_t W,
                     int32_t dtype, void *workspace, uint64_t workspace_bytes, void *stream,
                     int32_t *device_status_or_null);

/*
 * Diagnostics (no counterpart on the page): the execution plan the library
 * would use for a shape, as text lines "key=value" (H-block split, channels
 * per thread, warps, whether the main kernel splits its registers by
 * warpgroup, rows per stage, ring depth, CTAs, shared memory,
 * workspace layout, reduce shape; per-H-block CTA and slot ranges as comma
 * lists). kind: MCC1D_PLAN_BWD (mcc1d_bwd, W = 3), MCC1D_PLAN_BWD_EX (the
 * strided calls, 1 <= W <= 8) or MCC1D_PLAN_FWD (mcc1d_fwd, 1 <= W <= 8; with a GPU the
 * forward's plan also depends on its kernel's register count). Writes at most
 * buf_bytes - 1 characters plus a terminating NUL to buf (buf may be NULL);
 * *needed_out (optional) receives the full length + 1. Host only; shape
 * errors as mcc1d_bwd_workspace_size, MCC1D_ERR_PARAM_INVALID for a bad kind.
 */
enum { MCC1D_PLAN_BWD = 0, MCC1D_PLAN_BWD_EX = 1, MCC1D_PLAN_FWD = 2 };
int32_t mcc1d_plan_describe(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype,
                            int32_t kind, char *buf, uint64_t buf_bytes, uint64_t *needed_out);

/*
 * Device check (no counterpart on the page). Every call that launches
 * compares the current device's SM count (cudaDevAttrMultiProcessorCount,
 * read once per device) with MCC1D_PLAN_SMS and refuses a smaller device with
 * MCC1D_ERR_DEVICE. mcc1d_check_sm_count applies that rule to a given count
 * (host only; MCC1D_OK or MCC1D_ERR_DEVICE). mcc1d_device_sm_count writes
 * the current device's count to *sm_count_out (MCC1D_ERR_PARAM_NULLPTR for a
 * null pointer, MCC1D_ERR_CUDA when the runtime cannot say).
 */
int32_t mcc1d_check_sm_count(int32_t sm_count);
int32_t mcc1d_device_sm_count(int32_t *sm_count_out);

/*
 * Self-test of the bounded device-side wait (no counterpart on the page).
 * Every wait inside the library's kernels gives up after about 2 s and turns
 * into MCC1D_ERR_DEVICE_TIMEOUT instead of hanging the GPU. This call runs
 * that same wait in one thread on `stream`: with arrive != 0 the thread
 * signals the barrier first and MCC1D_OK is written to *device_status; with
 * arrive == 0 nothing ever signals it, the wait runs out (about 2 s) and
 * MCC1D_ERR_DEVICE_TIMEOUT is written. The context stays usable afterwards.
 * device_status: a 4-byte-aligned device (or device-accessible) int32.
 * Asynchronous; MCC1D_ERR_PARAM_NULLPTR / MCC1D_ERR_PARAM_INVALID for a null
 * or misaligned pointer, MCC1D_ERR_CUDA if the launch fails.
 */
int32_t mcc1d_selftest_wait(int32_t *device_status, int32_t arrive, void *stream);

/* Static text for a status code; never NULL. */
const char *mcc1d_status_string(int32_t status);

/* Library version as major * 10000 + minor * 100 + patch. */
int32_t mcc1d_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MCC1D_H */
