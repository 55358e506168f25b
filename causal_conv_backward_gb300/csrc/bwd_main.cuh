// bwd_main.cuh - the backward's main kernel (producer warp + consumer warps)
// as templates over the element type, rows per stage, channels per thread
// and the kernel width W. kernels.cu instantiates W = 3, the width the
// operator page supports; kernels_w.cu instantiates the other widths of the
// strided entry points.
//
// Operation (CANN page "aclnnMaskedCausalConv1dBackward", 功能说明 / 计算公式),
// per channel h: gYm(i) = mask(i) * gradY(i); gradX(i) = sum_k gYm(i+k) w(W-1-k);
// gradWeight(k) = sum_{j,i} gYm(i+W-1-k) x(i); gYm zero for i >= S.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "plan.h"

namespace mcc1d {

constexpr int kMaxThreads = 288;                  // 8 consumer warps + producer

struct MainParams {
    const uint8_t *gy;     // [S,B,H] 16-bit elements, addressed in bytes
    const uint8_t *x;      // [S,B,H]
    const uint16_t *w;     // [W,H]
    const uint8_t *mask;   // [B,S] or null
    uint8_t *gx;           // [S,B,H]
    float *part;           // [nslots][W][hb_width]
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

// ------------------------------------------------------------------ producer
template <int R, int W>
__device__ __forceinline__ uint32_t stage_mask_byte(const MainParams &p, const Cursor &c, int lane)
{
    if (lane >= R + W - 1)
        return 0;
    const int64_t row = c.i + lane;
    if (row >= p.S)
        return 0;  // past the end of the sequence: zero padding
    if (p.mask == nullptr)
        return 1;
    return __ldg(p.mask + (int64_t)c.j * p.m_b + row * p.m_s) != 0 ? 1u : 0u;
}

// The bounded wait, out of line unless the kernel splits its registers.
template <int PT>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity)
{
    if constexpr (PT == kSplitProducerThreads)
        return mbar_wait_bounded_inline(bar, parity);
    else
        return mbar_wait_bounded(bar, parity);
}

template <int R, int W, int PT>
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
    uint32_t mnext = stage_mask_byte<R, W>(p, cur, lane);
    while (cur.pos < r1) {
        const int n = cur.rows<R>(p.S);
        const bool head = (stage == 0) || (cur.i == 0);
        const uint32_t mcur = mnext;
        if (stage >= NS) {
            const bool ok = wait_bounded<PT>(bar_empty0 + 8u * slot, ph ^ 1u);
            dead = __any_sync(0xFFFFFFFFu, !ok);
            if (dead)
                break;
        }
        if (lane < R + W - 1)
            smem[p.off_mask + 32u * slot + lane] = (uint8_t)mcur;
        {
            Cursor nx = cur;
            nx.advance(n, p.S, p.B);
            if (nx.pos < r1)
                mnext = stage_mask_byte<R, W>(p, nx, lane);
        }
        const int64_t hb0 = (int64_t)cur.hb * p.hb_width;
        const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
        const uint32_t wbytes = (uint32_t)width * 2u;
        const int q0 = head ? 0 : W - 1;       // first gradY slot row this stage loads
        int64_t q1 = (int64_t)n + W - 1;       // gradY slot rows [q0, q1) lie inside S
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
                bulk_g2s(slot_base + (uint32_t)(R + W - 1) * p.row_bytes, p.x + 2 * cur.i * p.x_s,
                         (uint32_t)n * wbytes, bar_full0 + 8u * slot);
            }
        } else if (lane < nG) {
            const int q = q0 + lane;
            const int64_t e = (cur.i + q) * p.gy_s + (int64_t)cur.j * p.gy_b + hb0;
            bulk_g2s(slot_base + (uint32_t)q * p.row_bytes, p.gy + 2 * e, wbytes, bar_full0 + 8u * slot);
        } else if (lane < nG + n) {
            const int q = lane - nG;
            const int64_t e = (cur.i + q) * p.x_s + (int64_t)cur.j * p.x_b + hb0;
            bulk_g2s(slot_base + (uint32_t)(R + W - 1 + q) * p.row_bytes, p.x + 2 * e, wbytes,
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
        if (!wait_bounded<PT>(bar_full0 + 8u * s, (uint32_t)((last / NS) & 1)))
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

// BS: gradX rows leave through the slot with bulk copies (4 KB rows over long
// CTA ranges) instead of per-thread streaming stores.
template <int DT, int R, int NP, int W, bool BS, int PT>
__device__ bool consume(const MainParams &p, uint8_t *smem, int64_t r0, int64_t r1, int ct, int lane)
{
    const int NS = p.stages;
    const int nct = (int)blockDim.x - PT;                          // consumer threads
    const uint32_t bar_full0 = smem_u32(smem + p.off_bar);
    const uint32_t bar_empty0 = bar_full0 + 8u * (uint32_t)NS;
    constexpr int CH = 2 * NP;                                     // channels per thread
    constexpr int WH = W - 1;                                      // rows of the window
    constexpr bool kStageSums = W <= 3;                            // per-stage gradWeight level
    // Wide kernels (kCertMinWBwd): gradX by a certified plain sum, the
    // cascade only where the certificate fails (see below).
    constexpr bool kCF = W >= kCertMinWBwd && !BS;
    constexpr float kCert = cert_factor<DT, W>();
    // the fallback finds the W-1 rows before a stage in the previous slot,
    // whose look-ahead holds R rows; one failure bit per (row, channel pair)
    static_assert(!kCF || W - 1 <= R, "certified sums need W - 1 <= R");
    static_assert(!kCF || R * NP <= 32, "one 32-bit failure mask per stage");
    float *outer = reinterpret_cast<float *>(smem + p.off_outer);  // [W*CH][nct]
    const int64_t row_stride = 2 * (int64_t)p.B * p.H;             // bytes from row i to i+1
    const int c = blockIdx.x;

    Cursor cur;
    cur.init(r0, r1, p.S, p.BS);
    int hb_cur = -1;
    bool active = false;
    Vf<NP> wt[W];                     // weight rows k = 0 .. W-1 of this thread's channels
    float2 mid[W][NP];
#pragma unroll
    for (int k = 0; k < W; ++k)
#pragma unroll
        for (int e = 0; e < NP; ++e)
            mid[k][e] = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < W * CH; ++q)
        outer[q * nct + ct] = 0.f;
    int since_flush = 0;
    Vf<NP> win[WH > 0 ? WH : 1];      // gYm(i) .. gYm(i+W-2) for the next row i
#pragma unroll
    for (int q = 0; q < (WH > 0 ? WH : 1); ++q)
#pragma unroll
        for (int e = 0; e < NP; ++e)
            win[q].e[e] = make_float2(0.f, 0.f);
    // certified sums: kCert * max_k |w_k| per channel, and sum |gYm| over the
    // window rows (both rounded up; the sum slides with the window and is
    // recomputed at every stage, so its rounding does not build up)
    float2 kmw[NP], gab[NP];
#pragma unroll
    for (int e = 0; e < NP; ++e)
        kmw[e] = gab[e] = make_float2(0.f, 0.f);

    // Writes this thread's share of the partial for H-block hb_cur and clears
    // the accumulators. Sum order: shared-memory level, then register level.
    auto flush_partial = [&]() {
        if (active) {
            const int64_t slot = p.slot_base[hb_cur] + (c - p.c_lo[hb_cur]);
            float *dst = p.part + slot * W * p.hb_width + CH * ct;
#pragma unroll
            for (int k = 0; k < W; ++k) {
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
        for (int k = 0; k < W; ++k)
#pragma unroll
            for (int e = 0; e < NP; ++e)
                mid[k][e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < W * CH; ++q)
            outer[q * nct + ct] = 0.f;
        since_flush = 0;
    };

    int slot = 0, stage = 0;
    uint32_t ph = 0;
    bool dead = false;
    int prev_slot = -1, n_prev = 0;
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
#pragma unroll
                for (int k = 0; k < W; ++k)
                    wt[k] = load_weight<DT, NP>(p, k, hb0 + CH * ct);
                if constexpr (kCF) {
#pragma unroll
                    for (int e = 0; e < NP; ++e) {
                        float mx = 0.f, my = 0.f;
#pragma unroll
                        for (int k = 0; k < W; ++k) {
                            mx = fmaxf(mx, fabsf(wt[k].e[e].x));
                            my = fmaxf(my, fabsf(wt[k].e[e].y));
                        }
                        kmw[e] = mul_ru(make_float2(kCert, kCert), make_float2(mx, my));
                    }
                }
            }
        }
        if (!dead) {
            const uint32_t bar = bar_full0 + 8u * slot;
            const bool ok = mbar_try_wait(bar, ph) || wait_bounded<PT>(bar, ph);
            dead = __any_sync(0xFFFFFFFFu, !ok);
        }
        if (!dead && active) {
            const uint8_t *sl = smem + (size_t)slot * p.slot_bytes + 2 * CH * ct;
            const uint8_t *gys = sl;                                   // gradY slot rows 0..R+W-2
            uint8_t *xs = const_cast<uint8_t *>(sl) + (size_t)(R + WH) * p.row_bytes;   // x slot rows 0..R-1
            const uint8_t *ms = smem + p.off_mask + 32u * slot;
            if (head) {
#pragma unroll
                for (int q = 0; q < WH; ++q)
                    win[q] = load_masked<DT, NP>(gys + (size_t)q * p.row_bytes, ms[q]);
            }
            if constexpr (kCF) {
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    float2 g = make_float2(0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < WH; ++q)
                        g = add_abs_ru(g, win[q].e[e]);
                    gab[e] = g;
                }
            }
            uint8_t *gxp = p.gx + 2 * (((cur.i * p.B + cur.j) * p.H) + (int64_t)hb_cur * p.hb_width + CH * ct);
            // gradWeight of this stage: W <= 3 sums the stage's R rows on
            // their own before adding them to the 16-stage level; wider
            // kernels add each row straight into that level, which frees
            // W*CH registers per thread (the sums keep the same three levels
            // otherwise: rows, 16-stage blocks, the whole CTA range).
            float2 in[W][NP];
#pragma unroll
            for (int k = 0; k < W; ++k)
#pragma unroll
                for (int e = 0; e < NP; ++e)
                    in[k][e] = make_float2(0.f, 0.f);
            float2 (&acc)[W][NP] = kStageSums ? in : mid;
            uint32_t fails = 0;
            // One row i+r: gradX from the window gYm(i+r .. i+r+W-2) and the
            // staged gradY row i+r+W-1; the W gradWeight taps against x(i+r).
            auto row = [&](int r) {
                const Vf<NP> gn = load_masked<DT, NP>(gys + (size_t)(r + WH) * p.row_bytes, ms[r + WH]);
                const Vf<NP> xv = unpack<DT, NP>(load_raw<NP>(xs + (size_t)r * p.row_bytes));
                uint32_t o[NP];
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    // gradX = sum_k gYm(i+k) w(W-1-k): exact fp32 products,
                    // a compensated sum, rounded once (sum_to16)
                    if constexpr (kCF) {
                        // plain sum s of the exact products in a depth-3
                        // tree; when kCert * max|w| * sum|gYm| (>= kCert *
                        // sum|products|, rounded up) <= |s|, round(s) is
                        // within 1 ulp of the exact sum rounded once
                        // (cert_factor); else the channel is recomputed
                        // after the stage
                        const float2 gr = add_abs_ru(gab[e], gn.e[e]);
                        const float2 sf = dot_tree<W>([&](int k) { return k < WH ? win[k].e[e] : gn.e[e]; },
                                                      [&](int k) { return wt[W - 1 - k].e[e]; });
                        const float2 lim = mul_ru(kmw[e], gr);
                        const bool ok = (lim.x <= fabsf(sf.x)) & (lim.y <= fabsf(sf.y));
                        o[e] = pack2<DT>(sf);
                        fails |= (ok ? 0u : 1u) << (r * NP + e);
                        gab[e] = sub_abs_ru(gr, win[0].e[e]);   // gYm(i+r) leaves the window
                    } else {
                        o[e] = sum_to16<DT, W>(
                            [&](int k) { return mul2(k < WH ? win[k].e[e] : gn.e[e], wt[W - 1 - k].e[e]); });
                    }
                    // gradWeight tap k pairs x(i) with gYm(i+W-1-k)
#pragma unroll
                    for (int k = 0; k < W; ++k)
                        acc[W - 1 - k][e] = fma2(k < WH ? win[k].e[e] : gn.e[e], xv.e[e], acc[W - 1 - k][e]);
                }
                if constexpr (BS) {
                    // x(i+r) was read from this slot row above and is dead
                    // now: the row takes gradX(i+r) instead
                    if constexpr (NP == 4)
                        *reinterpret_cast<uint4 *>(xs + (size_t)r * p.row_bytes) = make_uint4(o[0], o[1], o[2], o[3]);
                    else
                        *reinterpret_cast<uint2 *>(xs + (size_t)r * p.row_bytes) = make_uint2(o[0], o[1]);
                } else {
                    store_cs<NP>(gxp + (int64_t)r * row_stride, o);
                }
#pragma unroll
                for (int q = 0; q + 1 < WH; ++q)
                    win[q] = win[q + 1];
                if (WH > 0)
                    win[WH > 0 ? WH - 1 : 0] = gn;
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
            if constexpr (kCF) {
                // channels whose certificate failed (strong cancellation):
                // the cascade, from the staged rows, one failed (row,
                // channel pair) per iteration, each lane walking its own
                // bits; the rows before this stage are still in the previous
                // slot, which is released one stage late for this
                const uint8_t *psl = smem + (size_t)(prev_slot < 0 ? 0 : prev_slot) * p.slot_bytes + 2 * CH * ct;
                const uint8_t *pms = smem + p.off_mask + 32u * (prev_slot < 0 ? 0 : prev_slot);
                while (fails) {
                    const int b = __ffs(fails) - 1;
                    fails &= fails - 1;
                    const int r = b / NP, e = b % NP;
                    float2 qk[W];
#pragma unroll
                    for (int k = 0; k < W; ++k) {
                        const int q = r + k;
                        const bool here = head || q >= WH;
                        const uint8_t *rp = here ? gys + (size_t)q * p.row_bytes
                                                 : psl + (size_t)(n_prev + q) * p.row_bytes;
                        const uint8_t mb = here ? ms[q] : pms[n_prev + q];
                        qk[k] = mul2(load_masked_pair<DT>(rp + 4 * e, mb), pick_pair<NP>(wt[W - 1 - k], e));
                    }
                    const uint32_t v = sum_to16<DT, W>([&](int k) { return qk[k]; });
                    *reinterpret_cast<uint32_t *>(gxp + (int64_t)r * row_stride + 4 * e) = v;
                }
            }
            if constexpr (kStageSums) {
#pragma unroll
                for (int k = 0; k < W; ++k)
#pragma unroll
                    for (int e = 0; e < NP; ++e)
                        mid[k][e] = add2(mid[k][e], in[k][e]);
            }
            if (++since_flush == kFlushStages) {
#pragma unroll
                for (int k = 0; k < W; ++k)
#pragma unroll
                    for (int e = 0; e < NP; ++e) {
                        outer[(k * CH + 2 * e) * nct + ct] += mid[k][e].x;
                        outer[(k * CH + 2 * e + 1) * nct + ct] += mid[k][e].y;
                        mid[k][e] = make_float2(0.f, 0.f);
                    }
                since_flush = 0;
            }
        }
        if constexpr (BS) {
            // every consumer's gradX values of the stage are in the slot
            // (made visible to the bulk-copy engine); one thread stores the
            // rows and releases the slot once the copies have read it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("bar.sync 1, %0;" ::"r"(nct) : "memory");
            if (ct == 0 && !dead) {
                const int64_t hb0 = (int64_t)cur.hb * p.hb_width;
                const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
                const uint32_t xbase =
                    smem_u32(smem + (size_t)slot * p.slot_bytes) + (uint32_t)(R + WH) * p.row_bytes;
                for (int r = 0; r < n; ++r)
                    bulk_s2g(p.gx + 2 * (((cur.i + r) * p.B + cur.j) * p.H + hb0), xbase + (uint32_t)r * p.row_bytes,
                             (uint32_t)width * 2u);
                bulk_commit();
                bulk_wait_read_all();
                mbar_arrive(bar_empty0 + 8u * slot);
            }
        } else if constexpr (kCF) {
            // the previous slot stays readable until this stage's fallback is done
            __syncwarp();
            if (!dead && lane == 0 && prev_slot >= 0)
                mbar_arrive(bar_empty0 + 8u * prev_slot);
            prev_slot = slot;
            n_prev = n;
        } else {
            __syncwarp();
            if (!dead && lane == 0)
                mbar_arrive(bar_empty0 + 8u * slot);
        }
        cur.advance(n, p.S, p.B);
        ++stage;
        if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
        }
    }
    if (hb_cur >= 0)
        flush_partial();
    if constexpr (kCF) {
        __syncwarp();
        if (!dead && lane == 0 && prev_slot >= 0)
            mbar_arrive(bar_empty0 + 8u * prev_slot);
    }
    if (BS && ct == 0)
        bulk_wait_all();   // the gradX rows are written
    return dead;
}

// ------------------------------------------------------------------ kernels
template <int DT, int R, int NP, int W, bool BS, int PT = 32>
__device__ __forceinline__ void main_body(const MainParams &p)
{
    // one producer lane per staged row (R + W - 1 gradY rows, R x rows), and
    // the stage's mask bytes fit the slot's 32-byte mask record
    static_assert(2 * R + W - 1 <= 32, "a stage must not stage more rows than a warp has lanes");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_err;
    const int c = blockIdx.x;
    const int64_t r0 = cta_row_begin(c, p.N, p.ncta);
    const int64_t r1 = cta_row_begin(c + 1, p.N, p.ncta);
    const int consumer_warps = (int)((blockDim.x - PT) >> 5);
    if (threadIdx.x == 0) {
        s_err = 0;
        const uint32_t bar0 = smem_u32(smem + p.off_bar);
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bar0 + 8u * s, 1);                                    // full
            mbar_init(bar0 + 8u * (p.stages + s), BS ? 1u : (uint32_t)consumer_warps);  // empty
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // Launched as a programmatic dependent of whatever precedes it on the
    // stream (the previous call's reduce, typically): the set-up above may
    // overlap that kernel's tail, but no global memory is touched before it
    // has completed and its writes are visible. A no-op otherwise.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int lane = threadIdx.x & 31;
    bool dead = false;
    if (threadIdx.x < PT) {
        // the register split (PT = 128): the producer's warpgroup gives up
        // registers first, then the consumer warpgroups take them
        if constexpr (PT == kSplitProducerThreads)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSplitProducerRegs));
        if (threadIdx.x < 32)
            dead = produce<R, W, PT>(p, smem, r0, r1, lane);
    } else {
        if constexpr (PT == kSplitProducerThreads)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSplitConsumerRegs));
        dead = consume<DT, R, NP, W, BS, PT>(p, smem, r0, r1, (int)threadIdx.x - PT, lane);
    }
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

template <int DT, int R, int NP, int W, bool BS = false>
__global__ void __launch_bounds__(kMaxThreads) mcc1d_bwd_main(const __grid_constant__ MainParams p)
{
    main_body<DT, R, NP, W, BS>(p);
}

// The same kernel held to the registers that let two CTAs share an SM
// (65536 / (2 * 288) per thread), for the plans that run two per SM.
template <int DT, int R, int NP, int W>
__global__ void __launch_bounds__(kMaxThreads, 2) mcc1d_bwd_main_x2(const __grid_constant__ MainParams p)
{
    main_body<DT, R, NP, W, false>(p);
}

// The widest kernels with the register file split by warpgroup: the
// producer's warpgroup (one producing warp, three idle) at 56 registers, the
// consumer warpgroups at 224, from a launch at 168 per thread (384 threads).
template <int DT, int R, int NP, int W>
__global__ void __launch_bounds__(kSplitMaxThreads, 1) mcc1d_bwd_main_rs(const __grid_constant__ MainParams p)
{
    main_body<DT, R, NP, W, false, kSplitProducerThreads>(p);
}

typedef void (*MainFn)(MainParams);

}  // namespace mcc1d
