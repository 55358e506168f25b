// fwd.cu - sm_103a kernel of the masked causal depthwise conv1d forward.
//
// The forward of the operator whose gradient mcc1d_bwd computes (the CANN
// page "aclnnMaskedCausalConv1dBackward" names it MaskedCausalConv1d and
// calls the mask the convolution's output mask): for every channel h and
// kernel width W (3 on the page),
//   y(t,j) = mask(j,t) * sum_{k<W} w(k) * x(t-(W-1)+k, j)
//          (W = 3: w(0)*x(t-2) + w(1)*x(t-1) + w(2)*x(t))
// with x zero before t = 0. Transposing this map gives exactly the page's
// gradX and gradWeight formulas.
//
// Same streaming design as the backward, with the W-1-row halo behind each
// row instead of ahead: per stage the producer warp copies x rows t .. t+R-1
// into a ring slot with cp.async.bulk and stores the stage's output-mask
// bytes; consumer threads keep the last W-1 x rows in registers, form y with
// the compensated W-term sum and a streaming store. The halo rows
// t-(W-1) .. t-1 are real data only at the first stage of a CTA range that
// starts inside a sequence (at a sequence start they are the zero padding):
// they go to a separate W-1-row area once, so the slots hold output rows
// only and the ring holds more stages. With 4 KB rows the consumers write
// each y row back into the slot row it was read from and one thread stores
// the stage's rows with bulk copies (shared -> global), so y leaves in whole
// rows like x arrives; narrower rows keep per-thread streaming stores. No
// reduction, no workspace.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "device_common.cuh"
#include "device.h"
#include "launch.h"
#include "plan.h"

namespace mcc1d {

// Output rows per stage: 8 up to W = 3; wider kernels, bound by their
// per-stage work rather than HBM, take deeper stages (measured in one call
// against 8, 10, 12 and 16, and 20 and 24 from W = 6: W = 4, 5 best at 12;
// W >= 6 at 24 on H-blocks over 512 channels (`deep`), at 16 on narrower
// ones, where fewer consumer warps share the ring).
constexpr int fwd_rows(int W, bool deep)
{
    return W <= 3 ? 8 : W <= 5 ? 12 : deep ? 24 : 16;
}
constexpr int kFwdDeepMinHbWidth = 576;   // channels of an H-block that take deep stages
constexpr int kFwdMaxThreads = 288;  // 8 consumer warps + producer
constexpr int kFwdMaxStages = 8;
// 4 KB rows: two ring slots per CTA (more measured slower on this 1:1
// read/write stream), and over long CTA ranges y leaves by bulk copies
constexpr uint32_t kFwdWideRowBytes = 4096;
constexpr int kFwdWideMaxStages = 2;
constexpr int64_t kFwdBulkStoreMinRowsPerCta = 1024;

struct FwdParams {
    const uint8_t *x;      // [S,B,H] 16-bit, addressed in bytes
    const uint16_t *w;     // [W,H]
    const uint8_t *mask;   // [B,S] or null
    uint8_t *y;            // [S,B,H]
    int32_t *status;       // device word or null: set to kErrTimeout if a wait gives up
    int64_t S, BS, H, N;
    int32_t B, hb_width, ncta, stages;
    uint32_t row_bytes, slot_bytes, off_halo, off_mask, off_bar;
    int32_t contig_rows;
    // Input strides (elements; mask bytes); x has unit H stride and 16-byte
    // aligned rows (other layouts are gathered into a dense copy first).
    int64_t x_s, x_b, w_k, w_h, m_b, m_s;
    int32_t w_vec;         // weight rows can be read as aligned vectors
};

// Byte q of a stage (row cursor at output row t = c.i): q < W-1 says whether
// the halo row t-(W-1)+q exists (is >= 0); q >= W-1 is the output mask of row
// t+q-(W-1) (zero past the end of S).
template <int R, int W>
__device__ __forceinline__ uint32_t fwd_stage_byte(const FwdParams &p, const Cursor &c, int lane)
{
    if (lane < W - 1)
        return c.i - (W - 1) + lane >= 0 ? 1u : 0u;
    if (lane >= R + W - 1)
        return 0;
    const int64_t row = c.i + lane - (W - 1);
    if (row >= p.S)
        return 0;
    if (p.mask == nullptr)
        return 1;
    return __ldg(p.mask + (int64_t)c.j * p.m_b + row * p.m_s) != 0 ? 1u : 0u;
}

template <int R, int W>
__device__ bool fwd_produce(const FwdParams &p, uint8_t *smem, int64_t r0, int64_t r1, int lane)
{
    const int NS = p.stages;
    const uint32_t bar_full0 = smem_u32(smem + p.off_bar);
    const uint32_t bar_empty0 = bar_full0 + 8u * (uint32_t)NS;
    const uint32_t ring0 = smem_u32(smem);
    Cursor cur;
    cur.init(r0, r1, p.S, p.BS);
    int slot = 0, stage = 0;
    uint32_t ph = 0;
    bool dead = false;
    uint32_t mnext = fwd_stage_byte<R, W>(p, cur, lane);
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
        if (lane < R + W - 1)
            smem[p.off_mask + 32u * slot + lane] = (uint8_t)mcur;
        {
            Cursor nx = cur;
            nx.advance(n, p.S, p.B);
            if (nx.pos < r1)
                mnext = fwd_stage_byte<R, W>(p, nx, lane);
        }
        const int64_t hb0 = (int64_t)cur.hb * p.hb_width;
        const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
        const uint32_t wbytes = (uint32_t)width * 2u;
        // slot row r holds x row t+r (r < n); halo row q holds x row
        // t-(W-1)+q, loaded for q in [h0, W-1) at the first stage of a range
        // that starts inside a sequence, never again
        int h0 = W - 1;
        if (stage == 0 && cur.i > 0)
            h0 = cur.i >= W - 1 ? 0 : (int)(W - 1 - cur.i);
        const int nh = W - 1 - h0;
        __syncwarp();
        if (lane == 0)
            mbar_arrive_expect_tx(bar_full0 + 8u * slot, (uint32_t)(nh + n) * wbytes);
        __syncwarp();
        const uint32_t slot_base = ring0 + (uint32_t)slot * p.slot_bytes;
        const uint32_t halo_base = ring0 + p.off_halo;
        if (p.contig_rows) {
            if (lane == 0) {
                bulk_g2s(slot_base, p.x + 2 * cur.i * p.x_s, (uint32_t)n * wbytes, bar_full0 + 8u * slot);
                if (nh > 0)
                    bulk_g2s(halo_base + (uint32_t)h0 * p.row_bytes, p.x + 2 * (cur.i - (W - 1) + h0) * p.x_s,
                             (uint32_t)nh * wbytes, bar_full0 + 8u * slot);
            }
        } else if (lane < n) {
            const int64_t e = (cur.i + lane) * p.x_s + (int64_t)cur.j * p.x_b + hb0;
            bulk_g2s(slot_base + (uint32_t)lane * p.row_bytes, p.x + 2 * e, wbytes, bar_full0 + 8u * slot);
        } else if (lane < n + nh) {
            const int q = h0 + lane - n;
            const int64_t e = (cur.i - (W - 1) + q) * p.x_s + (int64_t)cur.j * p.x_b + hb0;
            bulk_g2s(halo_base + (uint32_t)q * p.row_bytes, p.x + 2 * e, wbytes, bar_full0 + 8u * slot);
        }
        cur.advance(n, p.S, p.B);
        ++stage;
        if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
        }
    }
    const int used = stage < NS ? stage : NS;
    for (int s = 0; s < used; ++s) {
        const int last = s + NS * ((stage - 1 - s) / NS);
        if (!mbar_wait_bounded(bar_full0 + 8u * s, (uint32_t)((last / NS) & 1)))
            dead = true;
    }
    return __any_sync(0xFFFFFFFFu, dead);
}

// Weight row k for channels h .. h + 2*NP - 1: one vector load when the rows
// are dense and aligned, else one 16-bit load per channel.
template <int DT, int NP>
__device__ __forceinline__ Vf<NP> fwd_weight(const FwdParams &p, int k, int64_t h)
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

template <int DT, int R, int NP, int W, bool BS>
__device__ bool fwd_consume(const FwdParams &p, uint8_t *smem, int64_t r0, int64_t r1, int ct, int lane)
{
    constexpr int CH = 2 * NP;
    constexpr int WH = W - 1;                  // rows of the window
    // Wide kernels: y by the backward's certified plain sum, the cascade
    // only for channels whose certificate fails, recomputed after the stage
    // from the staged rows (the slot keeps x rows: not with bulk stores).
    constexpr bool kCF = W >= kCertMinWFwd && !BS;
    constexpr float kCert = cert_factor<DT, W>();
    // the W-1 rows before a stage that follows a full stage are the previous
    // slot's last rows; one failure bit per (row, channel pair)
    static_assert(!kCF || W - 1 <= R, "certified sums need W - 1 <= R");
    static_assert(!kCF || R * NP <= 64, "one 64-bit failure mask per stage");
    // the stage's failure mask: one bit per (row, channel pair)
    using FailMask = typename std::conditional<(R * NP > 32), unsigned long long, uint32_t>::type;
    const int NS = p.stages;
    const uint32_t bar_full0 = smem_u32(smem + p.off_bar);
    const uint32_t bar_empty0 = bar_full0 + 8u * (uint32_t)NS;
    const int64_t row_stride = 2 * (int64_t)p.B * p.H;
    Cursor cur;
    cur.init(r0, r1, p.S, p.BS);
    int hb_cur = -1;
    bool active = false;
    Vf<NP> wt[W];                    // weight rows k = 0 .. W-1 of this thread's channels
    Vf<NP> win[WH > 0 ? WH : 1];     // x(t-(W-1)) .. x(t-1) for the next row t
#pragma unroll
    for (int q = 0; q < (WH > 0 ? WH : 1); ++q)
#pragma unroll
        for (int e = 0; e < NP; ++e)
            win[q].e[e] = make_float2(0.f, 0.f);
    // certified sums: kCert * max_k |w_k| per channel, and sum |x| over the
    // window rows (both rounded up; recomputed at every stage)
    float2 kmw[NP], gab[NP];
#pragma unroll
    for (int e = 0; e < NP; ++e)
        kmw[e] = gab[e] = make_float2(0.f, 0.f);
    int slot = 0, stage = 0;
    uint32_t ph = 0;
    bool dead = false;
    int prev_slot = -1, n_prev = 0;
    while (cur.pos < r1) {
        const int n = cur.rows<R>(p.S);
        const bool head = (stage == 0) || (cur.i == 0);
        if (cur.hb != hb_cur) {
            hb_cur = cur.hb;
            const int64_t hb0 = (int64_t)hb_cur * p.hb_width;
            const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
            active = CH * ct < width;
            if (active) {
#pragma unroll
                for (int k = 0; k < W; ++k)
                    wt[k] = fwd_weight<DT, NP>(p, k, hb0 + CH * ct);
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
            const bool ok = mbar_try_wait(bar, ph) || mbar_wait_bounded(bar, ph);
            dead = __any_sync(0xFFFFFFFFu, !ok);
        }
        if (!dead && active) {
            uint8_t *xs = smem + (size_t)slot * p.slot_bytes + 2 * CH * ct;
            const uint8_t *ms = smem + p.off_mask + 32u * slot;
            if (head) {
                // halo rows: staged at a range's first stage, zero (mask
                // byte 0) at a sequence start
                const uint8_t *hs = smem + p.off_halo + 2 * CH * ct;
#pragma unroll
                for (int q = 0; q < WH; ++q)
                    win[q] = load_masked<DT, NP>(hs + (size_t)q * p.row_bytes, ms[q]);
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
            uint8_t *yp = p.y + 2 * (((cur.i * p.B + cur.j) * p.H) + (int64_t)hb_cur * p.hb_width + CH * ct);
            FailMask fails = 0;
            auto row = [&](int r) {
                const Vf<NP> xn = unpack<DT, NP>(load_raw<NP>(xs + (size_t)r * p.row_bytes));
                const uint32_t keep = 0u - (uint32_t)ms[r + WH];
                uint32_t o[NP];
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    if constexpr (kCF) {
                        // plain sum of the exact products in a depth-3 tree,
                        // kept when kCert * max|w| * sum|x| (rounded up) <=
                        // |s| (within 1 ulp of the exact sum rounded once)
                        const float2 gr = add_abs_ru(gab[e], xn.e[e]);
                        const float2 sf = dot_tree<W>([&](int k) { return k < WH ? win[k].e[e] : xn.e[e]; },
                                                      [&](int k) { return wt[k].e[e]; });
                        const float2 lim = mul_ru(kmw[e], gr);
                        const bool ok = (lim.x <= fabsf(sf.x)) & (lim.y <= fabsf(sf.y));
                        o[e] = pack2<DT>(sf) & keep;
                        fails |= (FailMask)(ok ? 0u : 1u) << (r * NP + e);
                        gab[e] = sub_abs_ru(gr, win[0].e[e]);   // x(t+r-W+1) leaves the window
                    } else {
                        // exact fp32 products, summed and rounded once by
                        // sum_to16 (the backward's gradX sum)
                        o[e] = sum_to16<DT, W>(
                                   [&](int k) { return mul2(k < WH ? win[k].e[e] : xn.e[e], wt[k].e[e]); }) &
                               keep;  // output mask
                    }
                }
                if constexpr (BS) {
                    // x(t+r) was read from this slot row above and now lives
                    // in the register window: the row takes y(t+r) instead
                    if constexpr (NP == 4)
                        *reinterpret_cast<uint4 *>(xs + (size_t)r * p.row_bytes) = make_uint4(o[0], o[1], o[2], o[3]);
                    else
                        *reinterpret_cast<uint2 *>(xs + (size_t)r * p.row_bytes) = make_uint2(o[0], o[1]);
                } else {
                    store_cs<NP>(yp + (int64_t)r * row_stride, o);
                }
#pragma unroll
                for (int q = 0; q + 1 < WH; ++q)
                    win[q] = win[q + 1];
                if (WH > 0)
                    win[WH > 0 ? WH - 1 : 0] = xn;
            };
            if (n == R) {
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
                // failed channels (strong cancellation): the cascade over
                // x(t+r-W+1) .. x(t+r), one failed (row, channel pair) per
                // iteration, from this slot, the halo area at a head stage,
                // else the previous slot (released one stage late for
                // this); the stored value is overwritten
                const uint8_t *hs = smem + p.off_halo + 2 * CH * ct;
                const uint8_t *psl = smem + (size_t)(prev_slot < 0 ? 0 : prev_slot) * p.slot_bytes + 2 * CH * ct;
                while (fails) {
                    int b;
                    if constexpr (R * NP > 32)
                        b = __ffsll((long long)fails) - 1;
                    else
                        b = __ffs((int)fails) - 1;
                    fails &= fails - 1;
                    const int r = b / NP, e = b % NP;
                    float2 qk[W];
#pragma unroll
                    for (int k = 0; k < W; ++k) {
                        const int d = r + k - WH;   // x row relative to the stage's first
                        const uint8_t *rp = d >= 0 ? xs + (size_t)d * p.row_bytes
                                          : head   ? hs + (size_t)(WH + d) * p.row_bytes
                                                   : psl + (size_t)(n_prev + d) * p.row_bytes;
                        const uint8_t mb = (d < 0 && head) ? ms[WH + d] : (uint8_t)1;
                        qk[k] = mul2(load_masked_pair<DT>(rp + 4 * e, mb), pick_pair<NP>(wt[k], e));
                    }
                    const uint32_t keep = 0u - (uint32_t)ms[r + WH];
                    const uint32_t v = sum_to16<DT, W>([&](int k) { return qk[k]; }) & keep;
                    *reinterpret_cast<uint32_t *>(yp + (int64_t)r * row_stride + 4 * e) = v;
                }
            }
        }
        if constexpr (BS) {
            // every consumer's y values of the stage are in the slot (their
            // writes made visible to the bulk-copy engine); one thread stores
            // the rows, and releases the slot once the copies have read it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("bar.sync 1, %0;" ::"r"((int)blockDim.x - 32) : "memory");
            if (ct == 0 && !dead) {
                const int64_t hb0 = (int64_t)cur.hb * p.hb_width;
                const int64_t width = (p.H - hb0 < p.hb_width) ? (p.H - hb0) : p.hb_width;
                const uint32_t sbase = smem_u32(smem + (size_t)slot * p.slot_bytes);
                for (int r = 0; r < n; ++r)
                    bulk_s2g(p.y + 2 * (((cur.i + r) * p.B + cur.j) * p.H + hb0), sbase + (uint32_t)r * p.row_bytes,
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
    if constexpr (kCF) {
        __syncwarp();
        if (!dead && lane == 0 && prev_slot >= 0)
            mbar_arrive(bar_empty0 + 8u * prev_slot);
    }
    if (BS && ct == 0)
        bulk_wait_all();   // the y rows are written
    return dead;
}

template <int DT, int R, int NP, int W, bool BS>
__device__ __forceinline__ void fwd_body(const FwdParams &p)
{
    // one producer lane per staged row, and the stage's flag bytes fit the
    // slot's 32-byte record
    static_assert(R + W - 1 <= 32, "a stage must not stage more rows than a warp has lanes");
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
            mbar_init(bar0 + 8u * s, 1);
            mbar_init(bar0 + 8u * (p.stages + s), BS ? 1u : (uint32_t)consumer_warps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // a programmatic dependent of the preceding kernel: the set-up above may
    // overlap its tail; memory is touched only after it has completed. The
    // next kernel may start its own set-up now.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    bool dead;
    if (threadIdx.x < 32)
        dead = fwd_produce<R, W>(p, smem, r0, r1, lane);
    else
        dead = fwd_consume<DT, R, NP, W, BS>(p, smem, r0, r1, (int)threadIdx.x - 32, lane);
    if (dead && lane == 0)
        atomicOr(&s_err, 1);
    __syncthreads();
    if (threadIdx.x == 0 && s_err && p.status != nullptr)
        atomicOr(p.status, kErrTimeout);
}

// Held to the registers that let two CTAs share an SM (96), so the plan's
// register cap keeps two of them per SM.
template <int DT, int R, int NP, int W, bool BS>
__global__ void __launch_bounds__(kFwdMaxThreads, 2) mcc1d_fwd_main(const __grid_constant__ FwdParams p)
{
    fwd_body<DT, R, NP, W, BS>(p);
}

// The same kernel compiled for one CTA per SM, for the widest kernels, whose
// W weights and W-1 window rows per channel need the registers.
template <int DT, int R, int NP, int W>
__global__ void __launch_bounds__(kFwdMaxThreads, 1) mcc1d_fwd_main_1(const __grid_constant__ FwdParams p)
{
    fwd_body<DT, R, NP, W, false>(p);
}

typedef void (*FwdFn)(FwdParams);

// W = 3 (the page's width) with 8 or 4 channels per thread, its 4 KB rows
// (8 channels per thread) with bulk stores; other widths with 4 channels per
// thread (their plan keeps H-blocks of at most 1024 channels), from W = 6 in
// the one-CTA form.
template <int DT, int W>
static FwdFn fwd_pick(int vec, int variant)
{
    if constexpr (W == 3) {
        if (vec == 4)
            return variant != kFwdPlain ? nullptr : mcc1d_fwd_main<DT, fwd_rows(3, false), 2, 3, false>;
        return variant == kFwdBulkStores ? mcc1d_fwd_main<DT, fwd_rows(3, false), 4, 3, true>
             : variant == kFwdPlain      ? mcc1d_fwd_main<DT, fwd_rows(3, false), 4, 3, false>
                                         : nullptr;
    } else if constexpr (W >= 6) {
        if (vec != 4 || variant == kFwdBulkStores)
            return nullptr;
        return variant == kFwdDeep ? mcc1d_fwd_main_1<DT, fwd_rows(W, true), 2, W>
                                   : mcc1d_fwd_main_1<DT, fwd_rows(W, false), 2, W>;
    } else {
        return vec == 4 && variant == kFwdPlain ? mcc1d_fwd_main<DT, fwd_rows(W, false), 2, W, false> : nullptr;
    }
}

template <int DT>
static FwdFn fwd_pick_w(int vec, int W, int variant)
{
    switch (W) {
    case 1: return fwd_pick<DT, 1>(vec, variant);
    case 2: return fwd_pick<DT, 2>(vec, variant);
    case 3: return fwd_pick<DT, 3>(vec, variant);
    case 4: return fwd_pick<DT, 4>(vec, variant);
    case 5: return fwd_pick<DT, 5>(vec, variant);
    case 6: return fwd_pick<DT, 6>(vec, variant);
    case 7: return fwd_pick<DT, 7>(vec, variant);
    case 8: return fwd_pick<DT, 8>(vec, variant);
    default: return nullptr;
    }
}

static FwdFn fwd_kernel(int dtype, int vec, int W, int variant)
{
    return dtype == 0 ? fwd_pick_w<0>(vec, W, variant) : fwd_pick_w<1>(vec, W, variant);
}

bool fwd_bulk_store(const Plan &pl)
{
    return pl.W == 3 && pl.vec == 8 && pl.row_bytes >= kFwdWideRowBytes && long_ranges(pl) &&
           pl.rows_total / pl.ncta >= kFwdBulkStoreMinRowsPerCta;
}

int fwd_variant(const Plan &pl)
{
    if (fwd_bulk_store(pl))
        return kFwdBulkStores;
    return pl.W >= 6 && pl.hb_width >= kFwdDeepMinHbWidth ? kFwdDeep : kFwdPlain;
}

uint32_t fwd_ring_min_bytes(const Plan &pl)
{
    // as fwd_ring below with two slots
    const uint32_t slot = (uint32_t)fwd_rows(pl.W, fwd_variant(pl) == kFwdDeep) * pl.row_bytes;
    return 2u * (slot + 48u) + 64u + (uint32_t)(pl.W - 1) * pl.row_bytes;
}

FwdRing fwd_ring(const Plan &pl)
{
    // fwd_rows(W) output rows per slot, one W-1-row halo area; as many slots
    // as the CTA's share of shared memory allows, 2 .. kFwdMaxStages
    FwdRing r;
    r.rows_per_stage = fwd_rows(pl.W, fwd_variant(pl) == kFwdDeep);
    r.slot_bytes = (uint32_t)r.rows_per_stage * pl.row_bytes;
    const uint32_t halo_bytes = (uint32_t)(pl.W - 1) * pl.row_bytes;
    int64_t budget = kSmemPerSM / pl.ctas_per_sm - kSmemReservedPerCta;
    if (budget > kSmemDynMax)
        budget = kSmemDynMax;
    budget -= 64 + halo_bytes;
    int64_t ns = budget / (r.slot_bytes + 48);
    if (ns > kFwdMaxStages)
        ns = kFwdMaxStages;
    if (pl.row_bytes >= kFwdWideRowBytes && ns > kFwdWideMaxStages)
        ns = kFwdWideMaxStages;
    if (ns < 2)
        ns = 2;
    r.stages = (int32_t)ns;
    r.off_halo = (uint32_t)ns * r.slot_bytes;
    r.off_mask = r.off_halo + halo_bytes;
    r.off_bar = (r.off_mask + 32u * (uint32_t)ns + 15u) & ~15u;
    r.smem_bytes = r.off_bar + 16u * (uint32_t)ns;
    return r;
}

int fwd_kernel_regs(int dtype, int vec, int W, int variant)
{
    // registers per thread of the forward instance (cached per device and
    // instance; 0 when the runtime cannot say)
    static std::atomic<int> cache[64][12 * (kMaxW + 1)];
    if (W < 1 || W > kMaxW)
        return 0;
    const FwdFn fn = fwd_kernel(dtype, vec, W, variant);
    if (fn == nullptr)
        return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    const int slot = ((dtype * 2 + (vec == 4 ? 1 : 0)) * 3 + variant) * (kMaxW + 1) + W;
    std::atomic<int> &c = cache[dev & 63][slot];
    int r = c.load(std::memory_order_acquire);
    if (r > 0)
        return r;
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, reinterpret_cast<const void *>(fn)) != cudaSuccess)
        return 0;
    c.store(a.numRegs, std::memory_order_release);
    return a.numRegs;
}

int32_t launch_fwd(const Plan &pl, const Layout &L, const void *x, const void *weight, const uint8_t *mask,
                   void *y, int32_t *status, cudaStream_t stream)
{
    // Same CTA partition as the backward; the ring holds x rows only.
    FwdParams fp;
    fp.x = static_cast<const uint8_t *>(x);
    fp.w = static_cast<const uint16_t *>(weight);
    fp.mask = mask;
    fp.y = static_cast<uint8_t *>(y);
    fp.status = status;
    fp.S = pl.S;
    fp.BS = pl.B * pl.S;
    fp.H = pl.H;
    fp.N = pl.rows_total;
    fp.B = (int32_t)pl.B;
    fp.hb_width = pl.hb_width;
    fp.ncta = pl.ncta;
    fp.row_bytes = pl.row_bytes;
    const FwdRing ring = fwd_ring(pl);
    fp.slot_bytes = ring.slot_bytes;
    fp.off_halo = ring.off_halo;
    fp.stages = ring.stages;
    fp.off_mask = ring.off_mask;
    fp.off_bar = ring.off_bar;
    const uint32_t smem = ring.smem_bytes;
    fp.x_s = L.x[0];
    fp.x_b = L.x[1];
    fp.w_k = L.w[0];
    fp.w_h = L.w[1];
    fp.m_b = L.m[0];
    fp.m_s = L.m[1];
    fp.w_vec = (L.w[1] == 1 && (L.w[0] * 2) % 16 == 0 && ((uintptr_t)weight & 15u) == 0) ? 1 : 0;
    fp.contig_rows = (pl.B == 1 && pl.n_hb == 1 && L.x[0] == pl.H && !long_ranges(pl)) ? 1 : 0;

    const int variant = fwd_variant(pl);
    FwdFn fn = fwd_kernel(pl.dtype, pl.vec, pl.W, variant);
    if (fn == nullptr)
        return kErrCuda;
    // the shared-memory attribute, once per (instance, device, context): a
    // context created after a device reset starts without it
    static std::atomic<unsigned long long> done[12 * (kMaxW + 1)][64];
    const int slot_id = ((pl.dtype * 2 + (pl.vec == 4 ? 1 : 0)) * 3 + variant) * (kMaxW + 1) + pl.W;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return kErrCuda;
    const unsigned long long ctx = current_context_id();
    if (ctx == 0 || done[slot_id][dev].load(std::memory_order_acquire) != ctx) {
        if (cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemDynMax) != cudaSuccess)
            return kErrCuda;
        done[slot_id][dev].store(ctx != 0 ? ctx : current_context_id(), std::memory_order_release);
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.ncta);
    cfg.blockDim = dim3((unsigned)pl.threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fn, fp) != cudaSuccess)
        return kErrCuda;
    return kOk;
}

}  // namespace mcc1d
