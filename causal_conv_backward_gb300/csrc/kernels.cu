// kernels.cu - sm_103a kernels of the masked causal depthwise conv1d backward.
//
// Operation (CANN operator page "aclnnMaskedCausalConv1dBackward", 功能说明 /
// 计算公式), for every depthwise channel h and kernel width W (3 on the page):
//   gYm(i,j)      = mask(j,i) * gradY(i,j)
//   gradX(i,j)    = sum_{k<W} gYm(i+k,j) * w(W-1-k)
//                   (W = 3: gYm(i)*w(2) + gYm(i+1)*w(1) + gYm(i+2)*w(0))
//   gradWeight(k) = sum_{j,i} gYm(i+W-1-k,j) * x(i,j)
// with gYm zero for i >= S.
//
// The work is pure streaming: each element of gradY and x is read once and
// each element of gradX written once, at 12 flops per 6 bytes, so the bound is
// HBM bandwidth and there is no dense contraction for the tensor cores.
//
// mcc1d_bwd_main (persistent, one range of rows per CTA):
//   The rows (hb, j, i) - H-block, batch, sequence position, i fastest - are
//   split into ncta contiguous ranges. Warp 0 is the producer: it walks its
//   CTA's range in stages of R rows and, per stage, copies the R rows of x and
//   the R rows of gradY W-1 positions ahead (plus the first W-1 rows when a
//   sequence starts) into a ring slot with cp.async.bulk, completing on the
//   slot's "full" mbarrier; it also stores the stage's mask bytes in the slot.
//   The consumer warps own one 16-byte vector (8 channels) each (8 bytes,
//   4 channels, when that fills the warps better, as for H = 384), keep the last
//   W-1 masked gradY rows in registers, and per row form gradX with a
//   compensated W-term sum (exact fp32 products + TwoSum), store it with
//   a streaming 16-byte store, and accumulate the W gradWeight taps in
//   fp32. Each CTA writes one fp32 partial [W][H-block] per H-block it
//   touched into the workspace. The main kernel's templates live in
//   bwd_main.cuh; this file instantiates W = 3, kernels_w.cu the other widths.
// mcc1d_bwd_reduce (programmatic dependent launch):
//   Sums the partials of every gradWeight column in a fixed order (64 serial
//   slices over the CTAs, then a pairwise tree), rounds once to the 16-bit
//   type and folds the CTAs' status words into the workspace header.
//
// Every device-side wait is bounded (kWaitLimitNs); a CTA whose wait gives up
// stops, waits (bounded) for its own bulk copies to land and reports
// kErrTimeout through its status word instead of hanging.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "bwd_main.cuh"
#include "device.h"
#include "device_common.cuh"
#include "launch.h"
#include "plan.h"

namespace mcc1d {

struct ReduceParams {
    const float *part;
    const int32_t *status;
    int32_t *header;
    uint8_t *gw;           // [W,H]
    int64_t H;
    int32_t hb_width, ncta, nchunk, W;
    int32_t splits, lanes_log2;     // splits x (1 << lanes_log2) = kReduceThreads
    int32_t c_lo[kMaxHb], c_hi[kMaxHb], slot_base[kMaxHb];
};

template <int DT>
__global__ void __launch_bounds__(kReduceThreads) mcc1d_bwd_reduce(const __grid_constant__ ReduceParams p)
{
    __shared__ float4 red[kReduceThreads];   // [split][lane]
    // the next call's main kernel may start its set-up now; it waits for
    // this grid's completion before it touches memory
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lanes = 1 << p.lanes_log2;
    const int lane = threadIdx.x & (lanes - 1), split = threadIdx.x >> p.lanes_log2;
    const int b = blockIdx.x;
    const int chunk = b % p.nchunk;
    const int k = (b / p.nchunk) % p.W;
    const int hb = b / (p.nchunk * p.W);
    const int64_t hb0 = (int64_t)hb * p.hb_width;
    const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
    const int col = chunk * 4 * lanes + 4 * lane;
    // The H-block's partials are the contiguous slots [base, base + n);
    // split s sums the slice [s*n/S, (s+1)*n/S) in order.
    const int n = p.c_hi[hb] - p.c_lo[hb] + 1;
    const int sb = (int)((int64_t)split * n / p.splits);
    const int se = (int)((int64_t)(split + 1) * n / p.splits);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < width) {
        const float *src = p.part + (((int64_t)p.slot_base[hb] + sb) * p.W + k) * p.hb_width + col;
        const int64_t step = (int64_t)p.W * p.hb_width;
#pragma unroll 4
        for (int q = sb; q < se; ++q, src += step) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(src));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
    }
    red[threadIdx.x] = acc;
    __syncthreads();
    // Fixed pairwise tree over the splits.
    for (int s = p.splits / 2; s >= 1; s >>= 1) {
        if (split < s) {
            float4 a = red[threadIdx.x];
            const float4 o = red[threadIdx.x + s * lanes];
            a.x += o.x;
            a.y += o.y;
            a.z += o.z;
            a.w += o.w;
            red[threadIdx.x] = a;
        }
        __syncthreads();
    }
    if (split == 0 && col < width) {
        const float4 a = red[lane];
        const uint32_t lo = pack2<DT>(make_float2(a.x, a.y));
        const uint32_t hi = pack2<DT>(make_float2(a.z, a.w));
        *reinterpret_cast<uint2 *>(p.gw + 2 * ((int64_t)k * p.H + hb0 + col)) = make_uint2(lo, hi);
    }
    if (b == 0) {
        int any = 0;
        for (int cc = threadIdx.x; cc < p.ncta; cc += blockDim.x)
            any |= (p.status[cc] != kOk);
        any = __syncthreads_or(any);
        if (threadIdx.x == 0)
            p.header[0] = any ? kErrTimeout : kOk;
    }
}

// Gather of a strided [S,B,H] 16-bit tensor into dense rows, 8 channels
// (one 16-byte store) per thread and step.
__global__ void __launch_bounds__(256) mcc1d_pack(const uint16_t *src, int64_t s_s, int64_t s_b,
                                                  int64_t s_h, uint16_t *dst, int64_t S, int64_t B,
                                                  int64_t H)
{
    const int64_t per_row = H / 8;
    const int64_t groups = S * B * per_row;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t hv = g % per_row, row = g / per_row;
        const int64_t j = row % B, i = row / B;
        const uint16_t *sp = src + i * s_s + j * s_b + hv * 8 * s_h;
        uint32_t u[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            u[e] = (uint32_t)__ldg(sp + 2 * e * s_h) | ((uint32_t)__ldg(sp + (2 * e + 1) * s_h) << 16);
        *reinterpret_cast<uint4 *>(dst + row * H + hv * 8) = make_uint4(u[0], u[1], u[2], u[3]);
    }
}

// ------------------------------------------------------------------ host launch
typedef void (*ReduceFn)(ReduceParams);

template <int DT, int NP>
static MainFn main_for(int R, bool bulk)
{
    if (bulk) {
        // bulk gradX stores: 4 KB rows only, which take 8 channels per thread
        if constexpr (NP == 4) {
            switch (R) {
            case 4: return mcc1d_bwd_main<DT, 4, NP, 3, true>;
            case 6: return mcc1d_bwd_main<DT, 6, NP, 3, true>;
            case 8: return mcc1d_bwd_main<DT, 8, NP, 3, true>;
            default: return nullptr;
            }
        }
        return nullptr;
    }
    switch (R) {
    case 4: return mcc1d_bwd_main<DT, 4, NP, 3>;
    case 6: return mcc1d_bwd_main<DT, 6, NP, 3>;
    case 8: return mcc1d_bwd_main<DT, 8, NP, 3>;
    case 14:  // deep stages of narrow rows (4 channels per thread) only
        if constexpr (NP == 2)
            return mcc1d_bwd_main<DT, 14, NP, 3>;
        else
            return nullptr;
    default: return nullptr;
    }
}

// Instances for W != 3 live in kernels_w.cu.
MainFn main_kernel_other_w(int dtype, int vec, int W, int R, bool split);

static MainFn main_kernel(int dtype, int R, int vec, int W, bool bulk, bool split)
{
    if (W != 3)
        return bulk ? nullptr : main_kernel_other_w(dtype, vec, W, R, split);
    if (split)
        return nullptr;
    if (dtype == 0)
        return vec == 4 ? main_for<0, 2>(R, bulk) : main_for<0, 4>(R, bulk);
    return vec == 4 ? main_for<1, 2>(R, bulk) : main_for<1, 4>(R, bulk);
}

// A kernel that splits its registers by warpgroup (setmaxnreg) is launched
// only when the registers the CTA starts with cover what its warpgroups hold
// after the split: the consumers' increase draws on what the producer's
// warpgroup gives up, and would otherwise wait for registers that never come.
static bool split_fits(const void *fn, int threads)
{
    constexpr int kSlots = 16;
    static std::mutex mu;
    static const void *fns[kSlots];
    static int regs[kSlots];
    if (threads % kSplitProducerThreads != 0 || threads <= kSplitProducerThreads || threads > kSplitMaxThreads)
        return false;
    int r = -1;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < kSlots && fns[i]; ++i)
            if (fns[i] == fn)
                r = regs[i];
        if (r < 0) {
            cudaFuncAttributes fa;
            if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess)
                return false;
            r = fa.numRegs;
            for (int i = 0; i < kSlots; ++i)
                if (!fns[i]) {
                    fns[i] = fn;
                    regs[i] = r;
                    break;
                }
        }
    }
    const int64_t need = (int64_t)kSplitProducerThreads * kSplitProducerRegs +
                         (int64_t)(threads - kSplitProducerThreads) * kSplitConsumerRegs;
    return (int64_t)r * threads >= need;
}

// gradX leaves by bulk copies out of the ring on 4 KB rows (8 channels per
// thread, W = 3) over long CTA ranges: +1.3 % on the 512K-token workload;
// narrow rows and short ranges lose to the per-stage barrier and wait.
static bool bwd_bulk_store(const Plan &pl)
{
    return pl.W == 3 && pl.vec == 8 && pl.row_bytes >= 4096 && pl.rows_total / pl.ncta >= kWideMinRowsPerCta;
}

// cudaFuncSetAttribute once per (kernel, device, context): a context created
// after a device reset starts without the attribute.
static bool ensure_smem_attr(const void *fn)
{
    constexpr int kSlots = 128, kDevs = 64;
    static std::mutex mu;
    static const void *fns[kSlots];
    static unsigned long long ctx_of[kSlots][kDevs];   // context the attribute was set in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs)
        return false;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    int slot = -1;
    for (int i = 0; i < kSlots; ++i) {
        if (fns[i] == fn) {
            slot = i;
            break;
        }
        if (fns[i] == nullptr) {
            fns[i] = fn;
            slot = i;
            break;
        }
    }
    if (slot < 0)
        return false;
    if (ctx != 0 && ctx_of[slot][dev] == ctx)
        return true;
    // leave room for the kernel's few bytes of static shared memory
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemDynMax) != cudaSuccess)
        return false;
    // the call above makes the device's primary context current if none was
    ctx_of[slot][dev] = ctx != 0 ? ctx : current_context_id();
    return true;
}

int32_t launch_reduce(const Plan &pl, void *workspace, void *gradWeight, cudaStream_t stream)
{
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    ReduceParams rp;
    rp.part = reinterpret_cast<const float *>(ws + pl.ws_part_off);
    rp.status = reinterpret_cast<const int32_t *>(ws + pl.ws_status_off);
    rp.header = reinterpret_cast<int32_t *>(ws);
    rp.gw = static_cast<uint8_t *>(gradWeight);
    rp.H = pl.H;
    rp.hb_width = pl.hb_width;
    rp.ncta = pl.ncta;
    rp.nchunk = (pl.hb_width + 4 * pl.red_lanes - 1) / (4 * pl.red_lanes);
    rp.splits = pl.red_splits;
    rp.lanes_log2 = 0;
    while ((1 << rp.lanes_log2) < pl.red_lanes)
        ++rp.lanes_log2;
    rp.W = pl.W;
    for (int h = 0; h < kMaxHb; ++h) {
        rp.c_lo[h] = pl.c_lo[h];
        rp.c_hi[h] = pl.c_hi[h];
        rp.slot_base[h] = pl.slot_base[h];
    }
    ReduceFn rfn = pl.dtype == 0 ? mcc1d_bwd_reduce<0> : mcc1d_bwd_reduce<1>;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t rcfg = {};
    rcfg.gridDim = dim3((unsigned)pl.reduce_blocks);
    rcfg.blockDim = dim3(kReduceThreads);
    rcfg.dynamicSmemBytes = 0;
    rcfg.stream = stream;
    rcfg.attrs = attr;
    rcfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&rcfg, rfn, rp) != cudaSuccess)
        return kErrCuda;
    return kOk;
}

int32_t launch_pack(const void *src, const int64_t strides[3], void *dst, int64_t S, int64_t B,
                    int64_t H, cudaStream_t stream)
{
    // grid-stride gather: eight 256-thread CTAs per SM of the device
    int sms = current_device_sm_count();
    if (sms <= 0)
        sms = kNumSMs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms * 8));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    if (cudaLaunchKernelEx(&cfg, mcc1d_pack, static_cast<const uint16_t *>(src), strides[0], strides[1],
                           strides[2], static_cast<uint16_t *>(dst), S, B, H) != cudaSuccess)
        return kErrCuda;
    return kOk;
}

int32_t launch_bwd(const Plan &pl, const Layout &L, const void *gradY, const void *x,
                   const void *weight, const uint8_t *mask, void *gradX, void *gradWeight,
                   void *workspace, cudaStream_t stream)
{
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    MainParams mp;
    mp.gy = static_cast<const uint8_t *>(gradY);
    mp.x = static_cast<const uint8_t *>(x);
    mp.w = static_cast<const uint16_t *>(weight);
    mp.mask = mask;
    mp.gx = static_cast<uint8_t *>(gradX);
    mp.part = reinterpret_cast<float *>(ws + pl.ws_part_off);
    mp.status = reinterpret_cast<int32_t *>(ws + pl.ws_status_off);
    mp.S = pl.S;
    mp.BS = pl.B * pl.S;
    mp.H = pl.H;
    mp.N = pl.rows_total;
    mp.B = (int32_t)pl.B;
    mp.hb_width = pl.hb_width;
    mp.ncta = pl.ncta;
    mp.stages = pl.stages;
    mp.row_bytes = pl.row_bytes;
    mp.slot_bytes = pl.slot_bytes;
    mp.off_mask = pl.off_mask;
    mp.off_bar = pl.off_bar;
    mp.off_outer = pl.off_outer;
    for (int h = 0; h < kMaxHb; ++h) {
        mp.c_lo[h] = pl.c_lo[h];
        mp.slot_base[h] = pl.slot_base[h];
    }
    mp.gy_s = L.gy[0];
    mp.gy_b = L.gy[1];
    mp.x_s = L.x[0];
    mp.x_b = L.x[1];
    mp.w_k = L.w[0];
    mp.w_h = L.w[1];
    mp.m_b = L.m[0];
    mp.m_s = L.m[1];
    mp.contig_rows = (pl.B == 1 && pl.n_hb == 1 && L.gy[0] == pl.H && L.x[0] == pl.H && !long_ranges(pl)) ? 1 : 0;
    mp.w_vec = (L.w[1] == 1 && (L.w[0] * 2) % 16 == 0 && ((uintptr_t)weight & 15u) == 0) ? 1 : 0;

    const int R = pl.rows_per_stage;
    MainFn mfn = main_kernel(pl.dtype, R, pl.vec, pl.W, bwd_bulk_store(pl), pl.reg_split != 0);
    if (!mfn)
        return kErrCuda;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(mfn)))
        return kErrCuda;
    if (pl.reg_split && !split_fits(reinterpret_cast<const void *>(mfn), pl.threads))
        return kErrCuda;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.ncta);
    cfg.blockDim = dim3((unsigned)pl.threads);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = stream;
    // a programmatic dependent of the preceding kernel (the kernel waits for
    // it before touching memory)
    cudaLaunchAttribute cattr[1];
    cattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    cattr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = cattr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mfn, mp) != cudaSuccess)
        return kErrCuda;
    return launch_reduce(pl, workspace, gradWeight, stream);
}

}  // namespace mcc1d
