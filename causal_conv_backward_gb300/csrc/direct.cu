// direct.cu - the backward with tensors read and written in place wherever
// they live, page-locked host memory included (mcc1d_bwd_host).
//
// The computation is the backward's (CANN page "aclnnMaskedCausalConv1dBackward",
// 功能说明 / 计算公式): gYm = mask * gradY, gradX(i) = gYm(i) w(2) + gYm(i+1) w(1)
// + gYm(i+2) w(0), gradWeight(k) = sum gYm(i+2-k) x(i). When gradY, x and
// gradX sit in host memory the host link (about 0.2 TB/s each way on a GB300
// node, against 7 TB/s of HBM) bounds the call, so this kernel does not
// stage through shared memory: every thread owns one vector of channels,
// loads U rows ahead with plain loads, and stores gradX straight back. The
// link then carries the inputs in, gradX out and the kernel computes, all at
// once, with no staging buffers or copies.
//
// It uses the backward's plan: the same CTA ranges and the same partial
// slots, so the backward's reduce kernel finishes it unchanged. Inside a CTA
// the gradWeight sums are grouped per U rows instead of per ring stage, so
// gradWeight may differ from mcc1d_bwd's in the last bit; gradX is the same
// arithmetic element by element.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "launch.h"
#include "plan.h"

namespace mcc1d {

constexpr int kDirectU = 8;            // rows loaded ahead per step
constexpr int kDirectMaxThreads = 256;

struct DirectParams {
    const uint8_t *gy, *x;  // [S,B,H] 16-bit, any device-accessible memory
    const uint16_t *w;      // [3,H]
    const uint8_t *mask;    // [B,S] or null
    uint8_t *gx;            // [S,B,H]
    float *part;            // [nslots][3][hb_width], device memory
    int32_t *status;        // [ncta]
    int64_t S, BS, H, N;
    int32_t B, hb_width, ncta;
    int32_t c_lo[kMaxHb], slot_base[kMaxHb];
};

template <int DT, int NP, int U>
__global__ void __launch_bounds__(kDirectMaxThreads) mcc1d_bwd_direct(const __grid_constant__ DirectParams p)
{
    extern __shared__ __align__(16) uint8_t dsmem[];
    constexpr int CH = 2 * NP;
    const int c = blockIdx.x, ct = threadIdx.x, nct = blockDim.x;
    const int64_t r0 = cta_row_begin(c, p.N, p.ncta);
    const int64_t r1 = cta_row_begin(c + 1, p.N, p.ncta);
    float *outer = reinterpret_cast<float *>(dsmem);  // [3*CH][nct]
    const int64_t row_elems = (int64_t)p.B * p.H;

    Cursor cur;
    cur.init(r0, r1, p.S, p.BS);
    int hb_cur = -1;
    bool active = false;
    Vf<NP> w0, w1, w2, g0, g1;
    float2 mid[3][NP];
#pragma unroll
    for (int k = 0; k < 3; ++k)
#pragma unroll
        for (int e = 0; e < NP; ++e)
            mid[k][e] = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 3 * CH; ++q)
        outer[q * nct + ct] = 0.f;
#pragma unroll
    for (int e = 0; e < NP; ++e)
        g0.e[e] = g1.e[e] = make_float2(0.f, 0.f);
    int since_flush = 0, step = 0;

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

    // Packed gradY row `row` of batch j (zero past the end of S) and its mask
    // word (all ones to keep, zero to drop, zero past the end of S).
    auto gy_raw = [&](int64_t row, int32_t j, int64_t h, uint32_t &keep) -> Raw<NP> {
        Raw<NP> r;
        if (row < p.S) {
            r = load_raw<NP>(p.gy + 2 * (row * row_elems + (int64_t)j * p.H + h));
            keep = (p.mask == nullptr || p.mask[(int64_t)j * p.S + row] != 0) ? 0xFFFFFFFFu : 0u;
        } else {
#pragma unroll
            for (int e = 0; e < NP; ++e)
                r.u[e] = 0u;
            keep = 0u;
        }
        return r;
    };
    auto masked = [&](Raw<NP> r, uint32_t keep) -> Vf<NP> {
#pragma unroll
        for (int e = 0; e < NP; ++e)
            r.u[e] &= keep;
        return unpack<DT, NP>(r);
    };

    while (cur.pos < r1) {
        const int n = cur.rows<U>(p.S);
        const bool head = (step == 0) || (cur.i == 0);
        const int64_t hb0 = (int64_t)cur.hb * p.hb_width;
        if (cur.hb != hb_cur) {
            if (hb_cur >= 0)
                flush_partial();
            hb_cur = cur.hb;
            const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
            active = CH * ct < width;
            if (active) {
                w0 = unpack<DT, NP>(load_raw<NP>(p.w + 0 * p.H + hb0 + CH * ct));
                w1 = unpack<DT, NP>(load_raw<NP>(p.w + 1 * p.H + hb0 + CH * ct));
                w2 = unpack<DT, NP>(load_raw<NP>(p.w + 2 * p.H + hb0 + CH * ct));
            }
        }
        if (active) {
            const int64_t h = hb0 + CH * ct;
            if (head) {
                uint32_t k0, k1;
                const Raw<NP> a = gy_raw(cur.i, cur.j, h, k0);
                const Raw<NP> b = gy_raw(cur.i + 1, cur.j, h, k1);
                g0 = masked(a, k0);
                g1 = masked(b, k1);
            }
            // issue every load of the step before using any of them
            Raw<NP> gq[U], xq[U];
            uint32_t kq[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (u < n) {
                    gq[u] = gy_raw(cur.i + u + 2, cur.j, h, kq[u]);
                    xq[u] = load_raw<NP>(p.x + 2 * ((cur.i + u) * row_elems + (int64_t)cur.j * p.H + h));
                }
            }
            float2 in[3][NP];
#pragma unroll
            for (int k = 0; k < 3; ++k)
#pragma unroll
                for (int e = 0; e < NP; ++e)
                    in[k][e] = make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (u < n) {
                    const Vf<NP> g2 = masked(gq[u], kq[u]);
                    const Vf<NP> xv = unpack<DT, NP>(xq[u]);
                    uint32_t o[NP];
#pragma unroll
                    for (int e = 0; e < NP; ++e) {
                        // the backward's gradX sum (exact products, TwoSum, one add,
                        // correction) and its three gradWeight taps
                        const float2 p0 = mul2(g0.e[e], w2.e[e]);
                        const float2 p1 = mul2(g1.e[e], w1.e[e]);
                        const float2 p2 = mul2(g2.e[e], w0.e[e]);
                        const float2 s = add2(p0, p1);
                        const float2 bb = sub2(s, p0);
                        const float2 err = add2(sub2(p0, sub2(s, bb)), sub2(p1, bb));
                        const float2 t = add2(s, p2);
                        o[e] = pack2<DT>(add2(t, err));
                        in[2][e] = fma2(g0.e[e], xv.e[e], in[2][e]);
                        in[1][e] = fma2(g1.e[e], xv.e[e], in[1][e]);
                        in[0][e] = fma2(g2.e[e], xv.e[e], in[0][e]);
                    }
                    uint8_t *dst = p.gx + 2 * ((cur.i + u) * row_elems + (int64_t)cur.j * p.H + h);
                    if (NP == 4)
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
                    else
                        *reinterpret_cast<uint2 *>(dst) = make_uint2(o[0], o[1]);
                    g0 = g1;
                    g1 = g2;
                }
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
        cur.advance(n, p.S, p.B);
        ++step;
    }
    if (hb_cur >= 0)
        flush_partial();
    if (ct == 0)
        p.status[c] = kOk;
    __threadfence();
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

typedef void (*DirectFn)(DirectParams);

int32_t launch_direct(const Plan &pl, const void *gradY, const void *x, const void *weight,
                      const uint8_t *mask, void *gradX, void *gradWeight, void *workspace,
                      cudaStream_t stream)
{
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    DirectParams dp;
    dp.gy = static_cast<const uint8_t *>(gradY);
    dp.x = static_cast<const uint8_t *>(x);
    dp.w = static_cast<const uint16_t *>(weight);
    dp.mask = mask;
    dp.gx = static_cast<uint8_t *>(gradX);
    dp.part = reinterpret_cast<float *>(ws + pl.ws_part_off);
    dp.status = reinterpret_cast<int32_t *>(ws + pl.ws_status_off);
    dp.S = pl.S;
    dp.BS = pl.B * pl.S;
    dp.H = pl.H;
    dp.N = pl.rows_total;
    dp.B = (int32_t)pl.B;
    dp.hb_width = pl.hb_width;
    dp.ncta = pl.ncta;
    for (int h = 0; h < kMaxHb; ++h) {
        dp.c_lo[h] = pl.c_lo[h];
        dp.slot_base[h] = pl.slot_base[h];
    }
    const int nct = pl.consumer_warps * 32;
    DirectFn fn;
    if (pl.dtype == 0)
        fn = pl.vec == 4 ? mcc1d_bwd_direct<0, 2, kDirectU> : mcc1d_bwd_direct<0, 4, kDirectU>;
    else
        fn = pl.vec == 4 ? mcc1d_bwd_direct<1, 2, kDirectU> : mcc1d_bwd_direct<1, 4, kDirectU>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.ncta);
    cfg.blockDim = dim3((unsigned)nct);
    cfg.dynamicSmemBytes = (size_t)3 * pl.vec * nct * sizeof(float);
    cfg.stream = stream;
    if (cudaLaunchKernelEx(&cfg, fn, dp) != cudaSuccess)
        return kErrCuda;
    return launch_reduce(pl, workspace, gradWeight, stream);
}

}  // namespace mcc1d
