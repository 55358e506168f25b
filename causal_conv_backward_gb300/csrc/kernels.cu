// kernels.cu - sm_103a kernels of the masked causal depthwise conv1d backward.
//
// Operation (CANN operator page "aclnnMaskedCausalConv1dBackward", 功能说明 /
// 计算公式), for every depthwise channel h:
//   gYm(i,j)      = mask(j,i) * gradY(i,j)
//   gradX(i,j)    = gYm(i,j)*w(2) + gYm(i+1,j)*w(1) + gYm(i+2,j)*w(0)
//   gradWeight(k) = sum_{j,i} gYm(i+2-k,j) * x(i,j)
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
//   the R rows of gradY two positions ahead (plus the first two rows when a
//   sequence starts) into a ring slot with cp.async.bulk, completing on the
//   slot's "full" mbarrier; it also stores the stage's mask bytes in the slot.
//   The consumer warps own one 16-byte vector (8 channels) each (8 bytes,
//   4 channels, when that fills the warps better, as for H = 384), keep the last
//   two masked gradY rows in registers, and per row form gradX with a
//   compensated three-term sum (exact fp32 products + TwoSum), store it with
//   a streaming 16-byte store, and accumulate the three gradWeight taps in
//   fp32. Each CTA writes one fp32 partial [3][H-block] per H-block it
//   touched into the workspace.
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

#include <atomic>

#include "device_common.cuh"
#include "launch.h"
#include "plan.h"

namespace mcc1d {

constexpr int kMaxThreads = 288;                  // 8 consumer warps + producer

struct MainParams {
    const uint8_t *gy;     // [S,B,H] 16-bit elements, addressed in bytes
    const uint8_t *x;      // [S,B,H]
    const uint16_t *w;     // [3,H]
    const uint8_t *mask;   // [B,S] or null
    uint8_t *gx;           // [S,B,H]
    float *part;           // [nslots][3][hb_width]
    int32_t *status;       // [ncta]
    int64_t S, BS, H, N;
    int32_t B, hb_width, ncta, stages;
    uint32_t row_bytes, slot_bytes, off_mask, off_bar, off_outer;
    int32_t c_lo[kMaxHb], slot_base[kMaxHb];
    // Input strides (elements; mask bytes). gradY and x have unit H stride.
    int64_t gy_s, gy_b, x_s, x_b, w_k, w_h, m_b, m_s;
    int32_t contig_rows;   // a stage's rows are adjacent in memory (one copy per tensor)
    int32_t w_vec;         // weight rows can be read as aligned vectors
};

struct ReduceParams {
    const float *part;
    const int32_t *status;
    int32_t *header;
    uint8_t *gw;           // [3,H]
    int64_t H;
    int32_t hb_width, ncta, nchunk;
    int32_t c_lo[kMaxHb], c_hi[kMaxHb], slot_base[kMaxHb];
};

// ------------------------------------------------------------------ producer
template <int R>
__device__ __forceinline__ uint32_t stage_mask_byte(const MainParams &p, const Cursor &c, int lane)
{
    if (lane >= R + 2)
        return 0;
    const int64_t row = c.i + lane;
    if (row >= p.S)
        return 0;  // past the end of the sequence: zero padding
    if (p.mask == nullptr)
        return 1;
    return __ldg(p.mask + (int64_t)c.j * p.m_b + row * p.m_s) != 0 ? 1u : 0u;
}

template <int R>
__device__ bool produce(const MainParams &p, uint8_t *smem, int64_t r0, int64_t r1, int lane)
{
    const int NS = p.stages;
    const uint32_t bar_full0 = smem_u32(smem + p.off_bar);
    const uint32_t bar_empty0 = bar_full0 + 8u * (uint32_t)NS;
    const uint32_t ring0 = smem_u32(smem);
    const bool contiguous = p.contig_rows != 0;

    Cursor cur;
    cur.init(r0, r1, p.S, p.BS);
    int slot = 0, stage = 0;
    uint32_t ph = 0;
    bool dead = false;
    uint32_t mnext = stage_mask_byte<R>(p, cur, lane);
    while (cur.pos < r1) {
        const int n = cur.rows<R>(p.S);
        const bool head = (stage == 0) || (cur.i == 0);
        const uint32_t mcur = mnext;
        if (stage >= NS) {
            const bool ok = mbar_wait_bounded(bar_empty0 + 8u * slot, ph ^ 1u);
            dead = __any_sync(0xFFFFFFFFu, !ok);
            if (dead)
                break;
        }
        if (lane < R + 2)
            smem[p.off_mask + 32u * slot + lane] = (uint8_t)mcur;
        {
            Cursor nx = cur;
            nx.advance(n, p.S, p.B);
            if (nx.pos < r1)
                mnext = stage_mask_byte<R>(p, nx, lane);
        }
        const int64_t hb0 = (int64_t)cur.hb * p.hb_width;
        const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
        const uint32_t wbytes = (uint32_t)width * 2u;
        const int q0 = head ? 0 : 2;           // first gradY slot row this stage loads
        int64_t q1 = (int64_t)n + 2;           // gradY slot rows [q0, q1) lie inside S
        if (p.S - cur.i < q1)
            q1 = p.S - cur.i;
        const int nG = q1 > q0 ? (int)(q1 - q0) : 0;
        __syncwarp();
        if (lane == 0)
            mbar_arrive_expect_tx(bar_full0 + 8u * slot, (uint32_t)(nG + n) * wbytes);
        __syncwarp();
        const uint32_t slot_base = ring0 + (uint32_t)slot * p.slot_bytes;
        if (contiguous) {
            // B = 1, one H-block and rows packed back to back: the stage's rows
            // are adjacent both in memory and in the slot, so one copy per
            // tensor moves them.
            if (lane == 0) {
                if (nG > 0)
                    bulk_g2s(slot_base + (uint32_t)q0 * p.row_bytes, p.gy + 2 * (cur.i + q0) * p.gy_s,
                             (uint32_t)nG * wbytes, bar_full0 + 8u * slot);
                bulk_g2s(slot_base + (uint32_t)(R + 2) * p.row_bytes, p.x + 2 * cur.i * p.x_s,
                         (uint32_t)n * wbytes, bar_full0 + 8u * slot);
            }
        } else if (lane < nG) {
            const int q = q0 + lane;
            const int64_t e = (cur.i + q) * p.gy_s + (int64_t)cur.j * p.gy_b + hb0;
            bulk_g2s(slot_base + (uint32_t)q * p.row_bytes, p.gy + 2 * e, wbytes, bar_full0 + 8u * slot);
        } else if (lane < nG + n) {
            const int q = lane - nG;
            const int64_t e = (cur.i + q) * p.x_s + (int64_t)cur.j * p.x_b + hb0;
            bulk_g2s(slot_base + (uint32_t)(R + 2 + q) * p.row_bytes, p.x + 2 * e, wbytes,
                     bar_full0 + 8u * slot);
        }
        cur.advance(n, p.S, p.B);
        ++stage;
        if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
        }
    }
    // Drain: every slot's last issued stage must have landed before the CTA
    // may exit (no-op in a normal run, where the consumers saw them all).
    const int used = stage < NS ? stage : NS;
    for (int s = 0; s < used; ++s) {
        const int last = s + NS * ((stage - 1 - s) / NS);
        if (!mbar_wait_bounded(bar_full0 + 8u * s, (uint32_t)((last / NS) & 1)))
            dead = true;
    }
    return __any_sync(0xFFFFFFFFu, dead);
}

// ------------------------------------------------------------------ consumers
// Weight taps k for channels h .. h + 2*NP - 1: one vector load when the
// weight rows are dense and aligned, else one 16-bit load per channel.
template <int DT, int NP>
__device__ __forceinline__ Vf<NP> load_weight(const MainParams &p, int k, int64_t h)
{
    if (p.w_vec)
        return unpack<DT, NP>(ldg_raw<NP>(p.w + k * p.w_k + h));
    Raw<NP> r;
#pragma unroll
    for (int e = 0; e < NP; ++e) {
        const uint32_t lo = __ldg(p.w + k * p.w_k + (h + 2 * e) * p.w_h);
        const uint32_t hi = __ldg(p.w + k * p.w_k + (h + 2 * e + 1) * p.w_h);
        r.u[e] = lo | (hi << 16);
    }
    return unpack<DT, NP>(r);
}

template <int DT, int R, int NP>
__device__ bool consume(const MainParams &p, uint8_t *smem, int64_t r0, int64_t r1, int ct, int lane)
{
    const int NS = p.stages;
    const int nct = (int)blockDim.x - 32;
    const uint32_t bar_full0 = smem_u32(smem + p.off_bar);
    const uint32_t bar_empty0 = bar_full0 + 8u * (uint32_t)NS;
    constexpr int CH = 2 * NP;                                     // channels per thread
    float *outer = reinterpret_cast<float *>(smem + p.off_outer);  // [3*CH][nct]
    const int64_t row_stride = 2 * (int64_t)p.B * p.H;             // bytes from row i to i+1
    const int c = blockIdx.x;

    Cursor cur;
    cur.init(r0, r1, p.S, p.BS);
    int hb_cur = -1;
    bool active = false;
    Vf<NP> w0, w1, w2;
    float2 mid[3][NP];
#pragma unroll
    for (int k = 0; k < 3; ++k)
#pragma unroll
        for (int e = 0; e < NP; ++e)
            mid[k][e] = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 3 * CH; ++q)
        outer[q * nct + ct] = 0.f;
    int since_flush = 0;
    Vf<NP> g0, g1;
#pragma unroll
    for (int e = 0; e < NP; ++e)
        g0.e[e] = g1.e[e] = make_float2(0.f, 0.f);

    // Writes this thread's share of the partial for H-block hb_cur and clears
    // the accumulators. Sum order: shared-memory level, then register level.
    auto flush_partial = [&]() {
        if (active) {
            const int64_t slot = p.slot_base[hb_cur] + (c - p.c_lo[hb_cur]);
            float *dst = p.part + slot * 3 * p.hb_width + CH * ct;
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                float v[CH];
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    v[2 * e] = outer[(k * CH + 2 * e) * nct + ct] + mid[k][e].x;
                    v[2 * e + 1] = outer[(k * CH + 2 * e + 1) * nct + ct] + mid[k][e].y;
                }
                float4 *d4 = reinterpret_cast<float4 *>(dst + (int64_t)k * p.hb_width);
#pragma unroll
                for (int q = 0; q < CH / 4; ++q)
                    d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
#pragma unroll
        for (int k = 0; k < 3; ++k)
#pragma unroll
            for (int e = 0; e < NP; ++e)
                mid[k][e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 3 * CH; ++q)
            outer[q * nct + ct] = 0.f;
        since_flush = 0;
    };

    int slot = 0, stage = 0;
    uint32_t ph = 0;
    bool dead = false;
    while (cur.pos < r1) {
        const int n = cur.rows<R>(p.S);
        const bool head = (stage == 0) || (cur.i == 0);
        if (cur.hb != hb_cur) {
            if (hb_cur >= 0)
                flush_partial();
            hb_cur = cur.hb;
            const int64_t hb0 = (int64_t)hb_cur * p.hb_width;
            const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
            active = CH * ct < width;
            if (active) {
                w0 = load_weight<DT, NP>(p, 0, hb0 + CH * ct);
                w1 = load_weight<DT, NP>(p, 1, hb0 + CH * ct);
                w2 = load_weight<DT, NP>(p, 2, hb0 + CH * ct);
            }
        }
        if (!dead) {
            const uint32_t bar = bar_full0 + 8u * slot;
            const bool ok = mbar_try_wait(bar, ph) || mbar_wait_bounded(bar, ph);
            dead = __any_sync(0xFFFFFFFFu, !ok);
        }
        if (!dead && active) {
            const uint8_t *sl = smem + (size_t)slot * p.slot_bytes + 2 * CH * ct;
            const uint8_t *gys = sl;                              // gradY slot rows 0..R+1
            const uint8_t *xs = sl + (size_t)(R + 2) * p.row_bytes;  // x slot rows 0..R-1
            const uint8_t *ms = smem + p.off_mask + 32u * slot;
            if (head) {
                g0 = load_masked<DT, NP>(gys, ms[0]);
                g1 = load_masked<DT, NP>(gys + p.row_bytes, ms[1]);
            }
            uint8_t *gxp = p.gx + 2 * (((cur.i * p.B + cur.j) * p.H) + (int64_t)hb_cur * p.hb_width + CH * ct);
            float2 in[3][NP];
#pragma unroll
            for (int k = 0; k < 3; ++k)
#pragma unroll
                for (int e = 0; e < NP; ++e)
                    in[k][e] = make_float2(0.f, 0.f);
            // One row: gradX(i+r) from the window (g0, g1) and the staged
            // gradY row i+r+2; the three gradWeight taps against x(i+r).
            auto row = [&](int r) {
                const Vf<NP> g2 = load_masked<DT, NP>(gys + (size_t)(r + 2) * p.row_bytes, ms[r + 2]);
                const Vf<NP> xv = unpack<DT, NP>(load_raw<NP>(xs + (size_t)r * p.row_bytes));
                uint32_t o[NP];
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    // gradX: products of two 16-bit values are exact in fp32;
                    // s + err == p0 + p1 exactly (TwoSum), then one more add
                    // and the correction: within a hair of the exact sum.
                    const float2 p0 = mul2(g0.e[e], w2.e[e]);
                    const float2 p1 = mul2(g1.e[e], w1.e[e]);
                    const float2 p2 = mul2(g2.e[e], w0.e[e]);
                    const float2 s = add2(p0, p1);
                    const float2 bb = sub2(s, p0);
                    const float2 err = add2(sub2(p0, sub2(s, bb)), sub2(p1, bb));
                    const float2 t = add2(s, p2);
                    o[e] = pack2<DT>(add2(t, err));
                    // gradWeight taps: k = 2 pairs x(i) with gYm(i), k = 1
                    // with gYm(i+1), k = 0 with gYm(i+2).
                    in[2][e] = fma2(g0.e[e], xv.e[e], in[2][e]);
                    in[1][e] = fma2(g1.e[e], xv.e[e], in[1][e]);
                    in[0][e] = fma2(g2.e[e], xv.e[e], in[0][e]);
                }
                store_cs<NP>(gxp + (int64_t)r * row_stride, o);
                g0 = g1;
                g1 = g2;
            };
            if (n == R) {
                // full stage: no per-row predicate, so the loads of all rows
                // can be issued ahead of the arithmetic
#pragma unroll
                for (int r = 0; r < R; ++r)
                    row(r);
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    if (r < n)
                        row(r);
            }
#pragma unroll
            for (int k = 0; k < 3; ++k)
#pragma unroll
                for (int e = 0; e < NP; ++e)
                    mid[k][e] = add2(mid[k][e], in[k][e]);
            if (++since_flush == kFlushStages) {
#pragma unroll
                for (int k = 0; k < 3; ++k)
#pragma unroll
                    for (int e = 0; e < NP; ++e) {
                        outer[(k * CH + 2 * e) * nct + ct] += mid[k][e].x;
                        outer[(k * CH + 2 * e + 1) * nct + ct] += mid[k][e].y;
                        mid[k][e] = make_float2(0.f, 0.f);
                    }
                since_flush = 0;
            }
        }
        __syncwarp();
        if (!dead && lane == 0)
            mbar_arrive(bar_empty0 + 8u * slot);
        cur.advance(n, p.S, p.B);
        ++stage;
        if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
        }
    }
    if (hb_cur >= 0)
        flush_partial();
    return dead;
}

// ------------------------------------------------------------------ kernels
template <int DT, int R, int NP>
__global__ void __launch_bounds__(kMaxThreads) mcc1d_bwd_main(const __grid_constant__ MainParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_err;
    const int c = blockIdx.x;
    const int64_t r0 = cta_row_begin(c, p.N, p.ncta);
    const int64_t r1 = cta_row_begin(c + 1, p.N, p.ncta);
    const int consumer_warps = (int)(blockDim.x >> 5) - 1;
    if (threadIdx.x == 0) {
        s_err = 0;
        const uint32_t bar0 = smem_u32(smem + p.off_bar);
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bar0 + 8u * s, 1);                                    // full
            mbar_init(bar0 + 8u * (p.stages + s), (uint32_t)consumer_warps);  // empty
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    bool dead;
    if (threadIdx.x < 32)
        dead = produce<R>(p, smem, r0, r1, lane);
    else
        dead = consume<DT, R, NP>(p, smem, r0, r1, (int)threadIdx.x - 32, lane);
    if (dead && lane == 0)
        atomicOr(&s_err, 1);
    __syncthreads();
    if (threadIdx.x == 0)
        p.status[c] = s_err ? kErrTimeout : kOk;
    // Only now let the reduce kernel be scheduled: every partial and status
    // word of this CTA is written and fenced before the trigger. (The reduce
    // also waits for this grid's completion before it reads them.)
    __threadfence();
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int DT>
__global__ void __launch_bounds__(kReduceSplits * kReduceLanes) mcc1d_bwd_reduce(const __grid_constant__ ReduceParams p)
{
    __shared__ float4 red[kReduceSplits][kReduceLanes];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x % kReduceLanes, split = threadIdx.x / kReduceLanes;
    const int b = blockIdx.x;
    const int chunk = b % p.nchunk;
    const int k = (b / p.nchunk) % 3;
    const int hb = b / (p.nchunk * 3);
    const int64_t hb0 = (int64_t)hb * p.hb_width;
    const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
    const int col = chunk * kReduceCols + 4 * lane;
    // The H-block's partials are the contiguous slots [base, base + n);
    // split s sums the slice [s*n/S, (s+1)*n/S) in order.
    const int n = p.c_hi[hb] - p.c_lo[hb] + 1;
    const int sb = (int)((int64_t)split * n / kReduceSplits);
    const int se = (int)((int64_t)(split + 1) * n / kReduceSplits);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < width) {
        const float *src = p.part + (((int64_t)p.slot_base[hb] + sb) * 3 + k) * p.hb_width + col;
        const int64_t step = 3 * (int64_t)p.hb_width;
#pragma unroll 4
        for (int q = sb; q < se; ++q, src += step) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(src));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
    }
    red[split][lane] = acc;
    __syncthreads();
    // Fixed pairwise tree over the splits.
#pragma unroll
    for (int s = kReduceSplits / 2; s >= 1; s >>= 1) {
        if (split < s) {
            float4 a = red[split][lane];
            const float4 o = red[split + s][lane];
            a.x += o.x;
            a.y += o.y;
            a.z += o.z;
            a.w += o.w;
            red[split][lane] = a;
        }
        __syncthreads();
    }
    if (split == 0 && col < width) {
        const float4 a = red[0][lane];
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
typedef void (*MainFn)(MainParams);
typedef void (*ReduceFn)(ReduceParams);

template <int DT, int NP>
static MainFn main_for(int R)
{
    switch (R) {
    case 4: return mcc1d_bwd_main<DT, 4, NP>;
    case 6: return mcc1d_bwd_main<DT, 6, NP>;
    case 8: return mcc1d_bwd_main<DT, 8, NP>;
    default: return nullptr;
    }
}

static MainFn main_kernel(int dtype, int R, int vec)
{
    if (dtype == 0)
        return vec == 4 ? main_for<0, 2>(R) : main_for<0, 4>(R);
    return vec == 4 ? main_for<1, 2>(R) : main_for<1, 4>(R);
}

// cudaFuncSetAttribute once per (kernel, device).
static bool ensure_smem_attr(const void *fn, int slot_id)
{
    static std::atomic<uint64_t> done[16];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    const uint64_t bit = 1ull << (dev & 63);
    if (done[slot_id].load(std::memory_order_acquire) & bit)
        return true;
    // leave room for the kernel's few bytes of static shared memory
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemPerCtaMax - 1024) != cudaSuccess)
        return false;
    done[slot_id].fetch_or(bit, std::memory_order_acq_rel);
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
    rp.nchunk = (pl.hb_width + kReduceCols - 1) / kReduceCols;
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
    rcfg.blockDim = dim3(kReduceSplits * kReduceLanes);
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(kNumSMs * 8));
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
    mp.contig_rows = (pl.B == 1 && pl.n_hb == 1 && L.gy[0] == pl.H && L.x[0] == pl.H) ? 1 : 0;
    mp.w_vec = (L.w[1] == 1 && (L.w[0] * 2) % 16 == 0 && ((uintptr_t)weight & 15u) == 0) ? 1 : 0;

    const int R = pl.rows_per_stage;
    MainFn mfn = main_kernel(pl.dtype, R, pl.vec);
    if (!mfn)
        return kErrCuda;
    const int attr_slot = (pl.dtype * 2 + (pl.vec == 4 ? 1 : 0)) * 4 + (R == 4 ? 0 : R == 6 ? 1 : 2);
    if (!ensure_smem_attr(reinterpret_cast<const void *>(mfn), attr_slot))
        return kErrCuda;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.ncta);
    cfg.blockDim = dim3((unsigned)pl.threads);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = stream;
    if (cudaLaunchKernelEx(&cfg, mfn, mp) != cudaSuccess)
        return kErrCuda;

    return launch_reduce(pl, workspace, gradWeight, stream);
}

}  // namespace mcc1d
