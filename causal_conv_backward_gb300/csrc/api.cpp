// api.cpp - the extern "C" entry points declared in include/mcc1d.h.
//
// Both phases validate in the order null pointers, dtype, shape, alignment,
// workspace; nothing touches a device before every check has passed.
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <string.h>

#include <string>

#include "device.h"
#include "launch.h"
#include "mcc1d.h"
#include "plan.h"

using namespace mcc1d;

// The forward needs about 96 registers a thread against the backward's 168,
// so it can keep more consumer warps resident per SM.
static constexpr int kFwdConsumerWarpsPerSM = 16;

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
    const int32_t dv = check_current_device();
    if (dv != kOk)
        return dv;
    return launch_bwd(p, dense_layout(S, B, H), gradY, x, weight, mask_or_null, gradX, gradWeight,
                      workspace, static_cast<cudaStream_t>(stream));
}

namespace {

// Device address of a pointer the current device can access: device memory,
// managed memory, or page-locked host memory. Null when it cannot.
void *device_address(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeUnregistered)
        return nullptr;
    int dev = -1;
    if (a.type == cudaMemoryTypeDevice && (cudaGetDevice(&dev) != cudaSuccess || dev != a.device))
        return nullptr;
    return a.devicePointer;
}

}  // namespace

extern "C" int32_t mcc1d_bwd_host(const void *gradY, const void *x, const void *weight,
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
    const int32_t dv = check_current_device();
    if (dv != kOk)
        return dv;
    const void *gy_d = device_address(gradY), *x_d = device_address(x), *w_d = device_address(weight);
    void *gx_d = device_address(gradX), *gw_d = device_address(gradWeight);
    const void *m_d = mask_or_null ? device_address(mask_or_null) : nullptr;
    if (!gy_d || !x_d || !w_d || !gx_d || !gw_d || (mask_or_null && !m_d))
        return kErrInvalid;
    return launch_direct(p, gy_d, x_d, w_d, static_cast<const uint8_t *>(m_d), gx_d, gw_d, workspace,
                         static_cast<cudaStream_t>(stream));
}

namespace {

// Plan of a strided call: which inputs are gathered into the workspace first,
// and where.
struct ExPlan {
    Plan plan;
    Layout L;          // layout the main kernel reads (dense for gathered inputs)
    Layout in;         // the caller's layout
    bool pack_gy, pack_x;
    uint64_t off_gy, off_x, bytes;
};

uint64_t round256(uint64_t v) { return (v + 255u) & ~(uint64_t)255u; }

// A 16-bit [S,B,H] input is streamed in place when its rows are contiguous
// along H and start on 16-byte boundaries.
bool streamable(const void *p, const int64_t st[3])
{
    return st[2] == 1 && ((uintptr_t)p & 15u) == 0 && (st[0] * 2) % 16 == 0 && (st[1] * 2) % 16 == 0;
}

int32_t make_ex(const mcc1d_tensors *t, int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype,
                ExPlan *e)
{
    if (!t || !t->gradY || !t->x || !t->weight || !t->gradX || !t->gradWeight)
        return kErrNull;
    const int32_t st = make_plan_general(S, B, H, W, dtype, &e->plan);
    if (st != kOk)
        return st;
    Layout in;
    const int64_t dims3[3] = {S, B, H};
    for (int d = 0; d < 3; ++d) {
        in.gy[d] = dims3[d] == 1 ? 0 : t->gradY_strides[d];
        in.x[d] = dims3[d] == 1 ? 0 : t->x_strides[d];
        if (t->gradY_strides[d] < 0 || t->x_strides[d] < 0)
            return kErrInvalid;
    }
    const int64_t dimsw[2] = {W, H}, dimsm[2] = {B, S};
    for (int d = 0; d < 2; ++d) {
        in.w[d] = dimsw[d] == 1 ? 0 : t->weight_strides[d];
        in.m[d] = dimsm[d] == 1 ? 0 : t->mask_strides[d];
        if (t->weight_strides[d] < 0 || (t->mask && t->mask_strides[d] < 0))
            return kErrInvalid;
    }
    if (((uintptr_t)t->gradY & 1u) || ((uintptr_t)t->x & 1u) || ((uintptr_t)t->weight & 1u) ||
        ((uintptr_t)t->gradX & 15u) || ((uintptr_t)t->gradWeight & 15u))
        return kErrInvalid;
    e->in = in;
    e->L = in;
    const uint64_t tensor_bytes = (uint64_t)S * (uint64_t)B * (uint64_t)H * 2u;
    e->pack_gy = !streamable(t->gradY, in.gy);
    e->pack_x = !streamable(t->x, in.x);
    const Layout dense = dense_layout(S, B, H);
    uint64_t off = round256(e->plan.ws_bytes);
    e->off_gy = e->off_x = 0;
    if (e->pack_gy) {
        e->off_gy = off;
        off = round256(off + tensor_bytes);
        for (int d = 0; d < 3; ++d)
            e->L.gy[d] = dense.gy[d];
    }
    if (e->pack_x) {
        e->off_x = off;
        off = round256(off + tensor_bytes);
        for (int d = 0; d < 3; ++d)
            e->L.x[d] = dense.x[d];
    }
    e->bytes = off;
    return kOk;
}

}  // namespace

extern "C" int32_t mcc1d_bwd_ex_workspace_size(const mcc1d_tensors *t, int64_t S, int64_t B,
                                               int64_t H, int64_t W, int32_t dtype,
                                               uint64_t *bytes_out)
{
    if (!bytes_out)
        return kErrNull;
    ExPlan e;
    const int32_t st = make_ex(t, S, B, H, W, dtype, &e);
    if (st != kOk)
        return st;
    *bytes_out = e.bytes;
    return kOk;
}

extern "C" int32_t mcc1d_bwd_ex(const mcc1d_tensors *t, int64_t S, int64_t B, int64_t H, int64_t W,
                                int32_t dtype, void *workspace, uint64_t workspace_bytes, void *stream)
{
    ExPlan e;
    const int32_t st = make_ex(t, S, B, H, W, dtype, &e);
    if (st != kOk)
        return st;
    if (!workspace)
        return kErrNull;
    if (!aligned16(workspace))
        return kErrInvalid;
    if (workspace_bytes < e.bytes)
        return kErrWorkspace;
    const int32_t dv = check_current_device();
    if (dv != kOk)
        return dv;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const void *gy = t->gradY, *x = t->x;
    if (e.pack_gy) {
        if (launch_pack(t->gradY, e.in.gy, ws + e.off_gy, S, B, H, s) != kOk)
            return kErrCuda;
        gy = ws + e.off_gy;
    }
    if (e.pack_x) {
        if (launch_pack(t->x, e.in.x, ws + e.off_x, S, B, H, s) != kOk)
            return kErrCuda;
        x = ws + e.off_x;
    }
    return launch_bwd(e.plan, e.L, gy, x, t->weight, t->mask, t->gradX, t->gradWeight, workspace, s);
}

namespace {

// The forward's plan. Its results do not depend on the CTA partition (no
// reduction), so the plan may use the compiled kernel's register count, asked
// of the runtime, to keep every CTA resident (no cap when the runtime cannot
// say, as on a machine without a GPU).
int32_t fwd_plan(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype, Plan *p)
{
    int32_t st = validate_shape_w(S, B, H, W, dtype);
    if (st != kOk)
        return st;
    // W = 3: blocks of up to 2048 channels, 8 or 4 per thread; other widths
    // keep their W weights and W-1 window rows per channel in registers with
    // 4 channels per thread and blocks of up to 1024 channels
    PlanOpts o = {kFwdConsumerWarpsPerSM, W == 3 ? kHbWidthWide : kHbWidthNarrow, 0, 8, true};
    st = make_plan_for(S, B, H, W, dtype, o, p);
    if (st != kOk)
        return st;
    // then CTAs per SM within the kernel's registers (as the runtime reports
    // them) and within shared memory for its smallest ring (two slots)
    o.regs_bound = fwd_kernel_regs(p->dtype, p->vec, p->W, fwd_variant(*p));
    o.smem_min_per_cta = (int)fwd_ring_min_bytes(*p);
    return make_plan_for(S, B, H, W, dtype, o, p);
}

}  // namespace

extern "C" int32_t mcc1d_fwd(const void *x, const void *weight, const uint8_t *mask_or_null, void *y,
                             void *stream, int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype,
                             int32_t *device_status_or_null)
{
    if (!x || !weight || !y)
        return kErrNull;
    int32_t st = validate_shape_w(S, B, H, W, dtype);
    if (st != kOk)
        return st;
    if (!aligned16(x) || !aligned16(weight) || !aligned16(y))
        return kErrInvalid;
    st = check_current_device();
    if (st != kOk)
        return st;
    Plan p;
    st = fwd_plan(S, B, H, W, dtype, &p);
    if (st != kOk)
        return st;
    return launch_fwd(p, dense_layout(S, B, H), x, weight, mask_or_null, y, device_status_or_null,
                      static_cast<cudaStream_t>(stream));
}

namespace {

// Plan of a strided forward: whether x is gathered into the workspace first.
struct FwdExPlan {
    Layout L;          // layout the kernel reads (dense x when gathered)
    Layout in;         // the caller's layout
    bool pack_x;
    uint64_t bytes;
};

// Validation and layout of a strided forward call (no device work).
int32_t make_fwd_ex(const mcc1d_fwd_tensors *t, int64_t S, int64_t B, int64_t H, int64_t W,
                    int32_t dtype, FwdExPlan *e)
{
    if (!t || !t->x || !t->weight || !t->y)
        return kErrNull;
    const int32_t st = validate_shape_w(S, B, H, W, dtype);
    if (st != kOk)
        return st;
    Layout in = dense_layout(S, B, H);
    const int64_t dims3[3] = {S, B, H};
    for (int d = 0; d < 3; ++d) {
        if (t->x_strides[d] < 0)
            return kErrInvalid;
        in.x[d] = dims3[d] == 1 ? 0 : t->x_strides[d];
    }
    const int64_t dimsw[2] = {W, H}, dimsm[2] = {B, S};
    for (int d = 0; d < 2; ++d) {
        if (t->weight_strides[d] < 0 || (t->mask && t->mask_strides[d] < 0))
            return kErrInvalid;
        in.w[d] = dimsw[d] == 1 ? 0 : t->weight_strides[d];
        in.m[d] = dimsm[d] == 1 ? 0 : t->mask_strides[d];
    }
    if (((uintptr_t)t->x & 1u) || ((uintptr_t)t->weight & 1u) || !aligned16(t->y))
        return kErrInvalid;
    e->in = in;
    e->L = in;
    e->pack_x = !streamable(t->x, in.x);
    e->bytes = 0;
    if (e->pack_x) {
        const Layout dense = dense_layout(S, B, H);
        for (int d = 0; d < 3; ++d)
            e->L.x[d] = dense.x[d];
        e->bytes = round256((uint64_t)S * (uint64_t)B * (uint64_t)H * 2u);
    }
    return kOk;
}

}  // namespace

extern "C" int32_t mcc1d_fwd_ex_workspace_size(const mcc1d_fwd_tensors *t, int64_t S, int64_t B,
                                               int64_t H, int64_t W, int32_t dtype,
                                               uint64_t *bytes_out)
{
    if (!bytes_out)
        return kErrNull;
    FwdExPlan e;
    const int32_t st = make_fwd_ex(t, S, B, H, W, dtype, &e);
    if (st != kOk)
        return st;
    *bytes_out = e.bytes;
    return kOk;
}

extern "C" int32_t mcc1d_fwd_ex(const mcc1d_fwd_tensors *t, int64_t S, int64_t B, int64_t H, int64_t W,
                                int32_t dtype, void *workspace, uint64_t workspace_bytes, void *stream,
                                int32_t *device_status_or_null)
{
    FwdExPlan e;
    int32_t st = make_fwd_ex(t, S, B, H, W, dtype, &e);
    if (st != kOk)
        return st;
    if (e.bytes > 0) {
        if (!workspace)
            return kErrNull;
        if (!aligned16(workspace))
            return kErrInvalid;
        if (workspace_bytes < e.bytes)
            return kErrWorkspace;
    }
    st = check_current_device();
    if (st != kOk)
        return st;
    Plan p;
    st = fwd_plan(S, B, H, W, dtype, &p);
    if (st != kOk)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const void *x = t->x;
    if (e.pack_x) {
        if (launch_pack(t->x, e.in.x, workspace, S, B, H, s) != kOk)
            return kErrCuda;
        x = workspace;
    }
    return launch_fwd(p, e.L, x, t->weight, t->mask, t->y, device_status_or_null, s);
}

extern "C" int32_t mcc1d_plan_describe(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype,
                                       int32_t kind, char *buf, uint64_t buf_bytes, uint64_t *needed_out)
{
    Plan p;
    int32_t st;
    if (kind == MCC1D_PLAN_BWD)
        st = make_plan(S, B, H, W, dtype, &p);
    else if (kind == MCC1D_PLAN_BWD_EX)
        st = make_plan_general(S, B, H, W, dtype, &p);
    else if (kind == MCC1D_PLAN_FWD)
        st = fwd_plan(S, B, H, W, dtype, &p);
    else
        return kErrInvalid;
    if (st != kOk)
        return st;
    if (kind == MCC1D_PLAN_FWD) {
        // the forward sizes its own ring and has no workspace or reduce
        const FwdRing r = fwd_ring(p);
        p.rows_per_stage = r.rows_per_stage;
        p.stages = r.stages;
        p.slot_bytes = r.slot_bytes;
        p.off_mask = r.off_mask;
        p.off_bar = r.off_bar;
        p.off_outer = r.smem_bytes;
        p.smem_bytes = r.smem_bytes;
        p.nslots = 0;
        p.ws_part_off = 0;
        p.ws_bytes = 0;
        p.reduce_blocks = 0;
        p.red_splits = 0;
        p.red_lanes = 0;
    }
    std::string t;
    auto kv = [&t](const char *k, long long v) {
        t += k;
        t += '=';
        t += std::to_string(v);
        t += '\n';
    };
    auto arr = [&t, &p](const char *k, const int32_t *a) {
        t += k;
        t += '=';
        for (int h = 0; h < p.n_hb; ++h) {
            if (h)
                t += ',';
            t += std::to_string(a[h]);
        }
        t += '\n';
    };
    kv("S", p.S);
    kv("B", p.B);
    kv("H", p.H);
    kv("W", p.W);
    kv("dtype", p.dtype);
    kv("hb_width", p.hb_width);
    kv("n_hb", p.n_hb);
    kv("vec", p.vec);
    kv("consumer_warps", p.consumer_warps);
    kv("threads", p.threads);
    kv("rows_per_stage", p.rows_per_stage);
    kv("stages", p.stages);
    kv("ctas_per_sm", p.ctas_per_sm);
    kv("rows_total", p.rows_total);
    kv("ncta", p.ncta);
    kv("nslots", p.nslots);
    kv("row_bytes", p.row_bytes);
    kv("slot_bytes", p.slot_bytes);
    kv("off_mask", p.off_mask);
    kv("off_bar", p.off_bar);
    kv("off_outer", p.off_outer);
    kv("smem_bytes", p.smem_bytes);
    kv("ws_part_off", (long long)p.ws_part_off);
    kv("ws_bytes", (long long)p.ws_bytes);
    kv("reduce_blocks", p.reduce_blocks);
    kv("red_splits", p.red_splits);
    kv("red_lanes", p.red_lanes);
    kv("regs_bound", kind == MCC1D_PLAN_FWD ? 0 : bwd_regs_bound(W));
    kv("reg_split", p.reg_split);
    kv("long_ranges", long_ranges(p) ? 1 : 0);
    arr("c_lo", p.c_lo);
    arr("c_hi", p.c_hi);
    arr("slot_base", p.slot_base);
    if (needed_out)
        *needed_out = t.size() + 1;
    if (buf && buf_bytes > 0) {
        const size_t n = t.size() < buf_bytes - 1 ? t.size() : (size_t)(buf_bytes - 1);
        memcpy(buf, t.data(), n);
        buf[n] = '\0';
    }
    return kOk;
}

extern "C" int32_t mcc1d_selftest_wait(int32_t *device_status, int32_t arrive, void *stream)
{
    if (!device_status)
        return kErrNull;
    if (((uintptr_t)device_status & 3u) != 0)
        return kErrInvalid;
    return launch_wait_selftest(device_status, arrive, static_cast<cudaStream_t>(stream));
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

extern "C" int32_t mcc1d_check_sm_count(int32_t sm_count) { return check_sm_count(sm_count); }

extern "C" int32_t mcc1d_device_sm_count(int32_t *sm_count_out)
{
    if (!sm_count_out)
        return kErrNull;
    const int32_t n = current_device_sm_count();
    if (n <= 0)
        return kErrCuda;
    *sm_count_out = n;
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
    case kErrDevice: return "MCC1D_ERR_DEVICE: the current device has fewer SMs than the launch plans assume (152)";
    default: return "unknown mcc1d status";
    }
}

extern "C" int32_t mcc1d_version(void) { return 100; }
