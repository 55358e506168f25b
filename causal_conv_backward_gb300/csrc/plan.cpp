// plan.cpp - shape validation and the launch plan (host only, no CUDA).
#include "plan.h"

#include <string.h>

namespace mcc1d {

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
static int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Limits from the operator page's constraints (约束说明): B in [1,32],
// B*S in [1, 512K], H in [384, 24576] and a multiple of 64, W == 3; and the
// two 16-bit types of its parameter table (参数说明).
int32_t validate_shape(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype)
{
    if (dtype != 0 && dtype != 1)
        return kErrInvalid;
    if (W != kW)
        return kErrShape;
    return validate_shape_w(S, B, H, W, dtype);
}

// The same limits with any kernel width 1 <= W <= kMaxW.
int32_t validate_shape_w(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype)
{
    if (dtype != 0 && dtype != 1)
        return kErrInvalid;
    if (W < 1 || W > kMaxW)
        return kErrShape;
    if (B < 1 || B > 32 || S < 1 || S > 524288 || B * S > 524288)
        return kErrShape;
    if (H < 384 || H > 24576 || H % 64 != 0)
        return kErrShape;
    return kOk;
}

int32_t make_plan(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype, Plan *p)
{
    const int32_t st = validate_shape(S, B, H, W, dtype);
    if (st != kOk)
        return st;
    return make_plan_general(S, B, H, W, dtype, p);
}

int32_t make_plan_general(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype, Plan *p)
{
    // Wide kernels keep W accumulators per channel: 4 channels per thread
    // and 1024-channel blocks keep them in registers. Up to kTwoCtaMaxW they
    // fit the two-CTA register bound, and sixteen consumer warps per SM hide
    // the longer arithmetic of each row.
    if (W >= 4)
        return make_plan_for(S, B, H, W, dtype,
                             {W <= kTwoCtaMaxW ? 16 : 8, kHbWidthNarrow, bwd_regs_bound(W), 5, false,
                              bwd_reg_split(W)},
                             p);
    const int32_t st = make_plan_for(S, B, H, W, dtype, {8, kHbWidthWide, bwd_regs_bound(W), 5, false}, p);
    if (st != kOk || p->rows_total / p->ncta >= kWideMinRowsPerCta)
        return st;
    return make_plan_for(S, B, H, W, dtype, {8, kHbWidthNarrow, bwd_regs_bound(W), 5, false}, p);
}

int32_t make_plan_for(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype, const PlanOpts &o,
                      Plan *p)
{
    const int target_consumer_warps = o.target_consumer_warps;
    const int max_hb_width = o.max_hb_width;
    const int regs_bound = o.regs_bound;
    int32_t st = validate_shape_w(S, B, H, W, dtype);
    if (st != kOk)
        return st;
    memset(p, 0, sizeof(*p));
    p->S = S;
    p->B = B;
    p->H = H;
    p->W = (int32_t)W;
    p->dtype = dtype;

    // H-blocks: as few as possible of at most max_hb_width halves, balanced,
    // each a multiple of 64 halves so every staged row is a multiple of 128 bytes.
    p->n_hb = (int32_t)ceil_div(H, max_hb_width);
    p->hb_width = (int32_t)round_up(ceil_div(H, p->n_hb), 64);
    // Channels per consumer thread: 8 (16-byte vectors), or 4 (8-byte) within
    // o.vec4_max_warps consumer warps, either always (the forward: twice the
    // threads in flight per row, at about 70 registers against 96; H-blocks up to
    // 1024) or when that leaves a smaller share of the consumer lanes idle
    // (the backward, within 5 warps: H-blocks of 384, 576 and 640; wider
    // blocks would give up their second CTA per SM, which costs more than the
    // idle lanes).
    p->vec = 8;
    {
        const int64_t v8 = p->hb_width / 8, v4 = p->hb_width / 4;
        const int64_t w8 = ceil_div(v8, 32), w4 = ceil_div(v4, 32);
        const bool better_lanes = v4 * w8 > v8 * w4;   // v4 / (32 w4) > v8 / (32 w8)
        if (w4 <= o.vec4_max_warps && (o.vec4_always || better_lanes))
            p->vec = 4;
    }
    if (W >= 4)
        p->vec = 4;
    const int vectors = p->hb_width / p->vec;
    p->consumer_warps = (int32_t)ceil_div(vectors, 32);
    p->threads = 32 * (p->consumer_warps + 1);
    p->reg_split = (o.reg_split && p->consumer_warps >= kSplitMinConsumerWarps) ? 1 : 0;
    if (p->reg_split) {
        // whole consumer warpgroups behind the producer's warpgroup (the
        // extra warps own no channels)
        p->consumer_warps = (int32_t)round_up(p->consumer_warps, 4);
        p->threads = kSplitProducerThreads + 32 * p->consumer_warps;
    }

    // Aim for at least target_consumer_warps consumer warps per SM.
    int cps = (int)ceil_div(target_consumer_warps, p->consumer_warps);
    while (cps > 1 && cps * p->threads > 2048)
        --cps;
    // ... and no more CTAs than the register file holds: each of an SM's four
    // schedulers has 16384 registers, so at r registers per thread it keeps
    // 16384 / (32 r) warps. r is the bound the kernel is compiled under, so a
    // plan never asks for CTAs that would wait for a second wave.
    if (regs_bound > 0) {
        const int warps_per_sm = 4 * (16384 / (32 * regs_bound));
        while (cps > 1 && cps * (p->threads / 32) > warps_per_sm)
            --cps;
    }
    // ... and no more than the shared memory holds at the kernel's minimum
    if (o.smem_min_per_cta > 0)
        while (cps > 1 && (int64_t)cps * (o.smem_min_per_cta + kSmemReservedPerCta) > kSmemPerSM)
            --cps;
    p->ctas_per_sm = cps;

    p->row_bytes = (uint32_t)p->hb_width * 2u;
    const uint32_t outer_bytes = (uint32_t)p->consumer_warps * 32u * (uint32_t)W * (uint32_t)p->vec * 4u;
    int64_t budget = kSmemPerSM / cps - kSmemReservedPerCta;
    if (budget > kSmemDynMax)
        budget = kSmemDynMax;

    // Rows per stage and ring depth: the deepest R (fewer barrier round trips)
    // that still leaves a ring of three slots, else the last choice with what
    // fits. Widths other than 3 have one instance: R = 6, or 10 at W = 4..6
    // and 8 at W = 7, 8. Long CTA ranges copy one row per bulk copy (see
    // long_ranges()); narrow rows (4 channels per thread) then spend most of
    // the producer's time per stage, not per byte, so they take R = 14
    // (2R + W - 1 = 30 copies, one per producer lane).
    int64_t ncta_est = (int64_t)kNumSMs * cps;
    const int64_t rows_all = (int64_t)p->n_hb * B * S;
    if (ncta_est > ceil_div(rows_all, kMinRowsPerCta))
        ncta_est = ceil_div(rows_all, kMinRowsPerCta);
    const bool deep = W == 3 && p->vec == 4 && rows_all / ncta_est >= kDeepMinRowsPerCta;
    // (deeper stages measured faster for W = 4..6 (10 rows) and 7, 8 (8);
    // from W = 5 the certified gradX sum also rereads the W-1 window rows
    // from the previous stage's slot, which holds R look-ahead rows)
    const int r_w3[3] = {8, 6, 4}, r_deep[4] = {14, 8, 6, 4}, r_other[1] = {6}, r_w10[1] = {10}, r_w78[1] = {8};
    const int *r_choices = deep ? r_deep : W == 3 ? r_w3 : (W >= 4 && W <= 6) ? r_w10 : W >= 7 ? r_w78 : r_other;
    const int n_choices = deep ? 4 : W == 3 ? 3 : 1;
    p->rows_per_stage = 0;
    for (int t = 0; t < n_choices; ++t) {
        const int R = r_choices[t];
        const int64_t slot = (int64_t)(2 * R + W - 1) * p->row_bytes;
        int64_t ns = (budget - outer_bytes - 64) / (slot + 48);
        if (ns >= 3 || t == n_choices - 1) {
            if (ns > 6)
                ns = 6;
            if (ns < 2)
                ns = 2;
            p->rows_per_stage = R;
            p->stages = (int32_t)ns;
            p->slot_bytes = (uint32_t)slot;
            break;
        }
    }
    p->off_mask = (uint32_t)p->stages * p->slot_bytes;
    p->off_bar = (uint32_t)round_up(p->off_mask + 32u * (uint32_t)p->stages, 16);
    p->off_outer = (uint32_t)round_up(p->off_bar + 16u * (uint32_t)p->stages, 16);
    p->smem_bytes = p->off_outer + outer_bytes;

    // Persistent CTAs over contiguous row ranges.
    p->rows_total = (int64_t)p->n_hb * B * S;
    int64_t ncta = (int64_t)kNumSMs * cps;
    const int64_t by_rows = ceil_div(p->rows_total, kMinRowsPerCta);
    if (ncta > by_rows)
        ncta = by_rows;
    if (ncta < 1)
        ncta = 1;
    p->ncta = (int32_t)ncta;

    const int64_t bs = B * S;
    for (int hb = 0; hb < p->n_hb; ++hb) {
        p->c_lo[hb] = p->ncta;
        p->c_hi[hb] = -1;
    }
    for (int64_t c = 0; c < ncta; ++c) {
        const int64_t r0 = cta_row_begin(c, p->rows_total, ncta);
        const int64_t r1 = cta_row_begin(c + 1, p->rows_total, ncta);
        const int hb0 = (int)(r0 / bs), hb1 = (int)((r1 - 1) / bs);
        for (int hb = hb0; hb <= hb1; ++hb) {
            if (c < p->c_lo[hb])
                p->c_lo[hb] = (int32_t)c;
            if (c > p->c_hi[hb])
                p->c_hi[hb] = (int32_t)c;
        }
    }

    p->nslots = 0;
    for (int hb = 0; hb < p->n_hb; ++hb) {
        p->slot_base[hb] = p->nslots;
        p->nslots += p->c_hi[hb] - p->c_lo[hb] + 1;
    }

    p->ws_status_off = kHeaderBytes;
    p->ws_part_off = kHeaderBytes + (uint64_t)round_up(4 * ncta, 256);
    p->ws_bytes = p->ws_part_off + (uint64_t)p->nslots * (uint64_t)W * (uint64_t)p->hb_width * 4u;
    // Reduce: each CTA sums red_lanes float4 column groups of one tap over all
    // partial slots of an H-block, in red_splits contiguous slices (as many as
    // the slots allow, so no slice is empty on average) and then a fixed
    // pairwise tree over the slices.
    int max_slots = 1;
    for (int hb = 0; hb < p->n_hb; ++hb)
        if (p->c_hi[hb] - p->c_lo[hb] + 1 > max_slots)
            max_slots = p->c_hi[hb] - p->c_lo[hb] + 1;
    int splits = kReduceMinSplits;
    while (splits < kReduceMaxSplits && 2 * splits <= max_slots)
        splits *= 2;
    p->red_splits = splits;
    p->red_lanes = kReduceThreads / splits;
    p->reduce_blocks = (int32_t)(p->n_hb * W * ceil_div(p->hb_width, 4 * p->red_lanes));
    return kOk;
}

}  // namespace mcc1d
