// plan.h - shape validation and the launch plans (host only).
//
// The backward's plan is a pure function of (S, B, H, W, dtype): the partition
// of the work, the order of every floating-point sum and the workspace size
// never depend on the device it later runs on, so equal inputs give
// bitwise-equal outputs. The forward's plan may also use its kernel's register
// count as the runtime reports it: each of its outputs is one thread's sum,
// so its results do not depend on the partition.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define MCC1D_HD __host__ __device__
#else
#define MCC1D_HD
#endif

namespace mcc1d {

constexpr int kW = 3;                 // the only kernel width the operator page supports
constexpr int kMaxW = 8;              // widest kernel the strided entry points accept
constexpr int kTwoCtaMaxW = 4;        // widths 4 .. kTwoCtaMaxW run two CTAs per SM
constexpr int kRegsOneCta = 168;      // register bound of the main kernel (288 threads, one CTA)
constexpr int kRegsTwoCta = 96;       // ... and of its two-CTA form (mcc1d_bwd_main_x2)
// From W = kSplitMinW the backward's main kernel splits the register file by
// warpgroup (mcc1d_bwd_main_rs): launched at kSplitLaunchRegs per thread, the
// producer's warpgroup (kSplitProducerThreads threads, one warp of them
// producing) drops to kSplitProducerRegs and the consumer warpgroups rise to
// kSplitConsumerRegs. The consumers' share must come from what the producer
// group gives up: 128 * 56 + 256 * 224 = 384 * 168 exactly at the widest
// plan (8 consumer warps), less for narrower ones.
constexpr int kSplitMinW = 5;
constexpr int kSplitProducerThreads = 128;
constexpr int kSplitLaunchRegs = 168;
constexpr int kSplitProducerRegs = 56;
constexpr int kSplitConsumerRegs = 224;
constexpr int kSplitMaxThreads = 384;
// Only H-blocks that need more than one consumer warpgroup split: narrower
// ones (at most 512 channels) would pad to a whole warpgroup behind a
// 4-warp producer group and fit one CTA per SM instead of three.
constexpr int kSplitMinConsumerWarps = 5;
static_assert(kSplitProducerThreads * kSplitProducerRegs +
                      (kSplitMaxThreads - kSplitProducerThreads) * kSplitConsumerRegs <=
                  kSplitMaxThreads * kSplitLaunchRegs,
              "the register split must fit the launch's registers");
inline bool bwd_reg_split(int64_t W) { return W >= kSplitMinW; }
constexpr int kDeepMinRowsPerCta = 256;  // CTA range long enough for 14-row stages
constexpr int kNumSMs = 152;          // GB300: 2 dies x 76 SMs (MCC1D_PLAN_SMS; checked per device)
constexpr int kSmemPerSM = 233472;    // 228 KB of shared memory per SM
constexpr int kSmemPerCtaMax = 232448;// 227 KB opt-in maximum per CTA
constexpr int kSmemReservedPerCta = 1024;
// Dynamic shared memory a kernel may be given: the opt-in maximum less room
// for the kernels' few bytes of static shared memory. The launch attribute is
// set to this, and no plan budgets a CTA more.
constexpr int kSmemDynMax = kSmemPerCtaMax - 1024;
constexpr int kMaxHb = 64;            // upper bound on H-blocks recorded in a plan
constexpr int kHbWidthNarrow = 1024;  // halves per H-block: 2 KB rows
constexpr int kHbWidthWide = 2048;    // 4 KB rows, for long CTA ranges
constexpr int kWideMinRowsPerCta = 1024;
constexpr int kMinRowsPerCta = 16;    // below this a CTA is not worth its pipeline fill
constexpr int kFlushStages = 16;      // stages between register -> shared accumulator flushes
constexpr int kReduceThreads = 512;   // threads per reduce CTA: splits x float4 column groups
constexpr int kReduceMinSplits = 8;   // contiguous slices of a column's partials per reduce CTA:
constexpr int kReduceMaxSplits = 64;  // the largest power of two <= the slots of an H-block, in range
constexpr uint64_t kHeaderBytes = 256;

// Status codes, the same values as the public header.
enum : int32_t {
    kOk = 0,
    kErrNull = 161001,
    kErrInvalid = 161002,
    kErrShape = 561002,
    kErrWorkspace = 561003,
    kErrCuda = 561100,
    kErrTimeout = 561101,
    kErrDevice = 561102,
};

struct Plan {
    int64_t S, B, H;
    int32_t W;               // kernel width (taps)
    int32_t dtype;           // 0 bf16, 1 fp16
    // H is cut into n_hb blocks of hb_width halves (the last may be narrower).
    int32_t hb_width, n_hb;
    // CTA shape: warp 0 produces (bulk copies), consumer_warps compute; each
    // consumer thread owns `vec` consecutive channels (8: a 16-byte vector,
    // or 4: an 8-byte vector) of the H-block.
    int32_t vec;
    int32_t consumer_warps, threads;
    int32_t reg_split;       // 1: the main kernel splits its registers by warpgroup
    int32_t rows_per_stage;  // R: rows of x (and R+W-1 of gradY) per ring slot
    int32_t stages;          // ring slots
    int32_t ctas_per_sm;
    // Work: the rows (hb, j, i), flattened with i fastest, N = n_hb*B*S, are
    // split into ncta contiguous ranges [c*N/ncta, (c+1)*N/ncta).
    int64_t rows_total;
    int32_t ncta;
    int32_t c_lo[kMaxHb], c_hi[kMaxHb];  // CTAs whose range touches H-block hb
    // Partial slots: CTA c's partial for H-block hb is slot
    // slot_base[hb] + c - c_lo[hb]; the slots of one H-block are contiguous.
    int32_t slot_base[kMaxHb];
    int32_t nslots;
    // Shared memory layout (bytes from the dynamic smem base).
    uint32_t row_bytes;      // stride of one staged row = hb_width * 2
    uint32_t slot_bytes;     // (2R + W - 1) rows
    uint32_t off_mask;       // stages x 32 mask bytes
    uint32_t off_bar;        // 2 x stages mbarriers
    uint32_t off_outer;      // W * vec fp32 accumulators per consumer thread
    uint32_t smem_bytes;
    // Workspace layout: header | per-CTA status words | fp32 partials
    // [nslots][W][hb_width].
    uint64_t ws_status_off, ws_part_off, ws_bytes;
    // Reduce launch.
    int32_t reduce_blocks;
    int32_t red_splits, red_lanes;   // reduce CTA shape: red_splits x red_lanes = kReduceThreads
};

// Strides of the inputs in elements (the mask's in bytes), outermost first:
// gradY and x [S,B,H], weight [W,H], mask [B,S]. The dense layout is
// gradY/x (B*H, H, 1), weight (H, 1), mask (S, 1).
struct Layout {
    int64_t gy[3], x[3], w[2], m[2];
};

inline Layout dense_layout(int64_t S, int64_t B, int64_t H)
{
    Layout L;
    L.gy[0] = L.x[0] = B * H;
    L.gy[1] = L.x[1] = H;
    L.gy[2] = L.x[2] = 1;
    L.w[0] = H;
    L.w[1] = 1;
    L.m[0] = S;
    L.m[1] = 1;
    return L;
}

// Shape and dtype checks of the page's constraints (W == 3). Returns kOk,
// kErrInvalid (dtype) or kErrShape. validate_shape_w allows 1 <= W <= kMaxW.
int32_t validate_shape(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype);
int32_t validate_shape_w(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype);

// Fills *p for a valid shape; returns the validate_shape status otherwise.
// make_plan is the backward's plan: 8 consumer warps per SM (its register
// budget), and 4 KB H-block rows when every CTA range is long enough for the
// larger copies to pay, else 2 KB. make_plan_for takes those choices from a
// PlanOpts (the forward asks for 16 consumer warps and 4 KB rows).
int32_t make_plan(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype, Plan *p);
// The backward's plan for any width 1 <= W <= kMaxW (the strided entry points).
int32_t make_plan_general(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype, Plan *p);
// What a kernel asks of its plan.
struct PlanOpts {
    int target_consumer_warps;   // consumer warps per SM to aim for
    int max_hb_width;            // widest H-block (channels)
    int regs_bound;              // registers per thread the kernel is held to; CTAs per SM
                                 // never exceed what the register file holds (0: no cap)
    int vec4_max_warps;          // 4 channels per thread allowed up to this many consumer warps
    bool vec4_always;            // ... and taken whenever allowed (else only for better lane use)
    bool reg_split = false;      // producer warpgroup + whole consumer warpgroups (setmaxnreg)
    int smem_min_per_cta = 0;    // shared memory a CTA cannot run without; CTAs per SM capped to fit (0: none)
};
int32_t make_plan_for(int64_t S, int64_t B, int64_t H, int64_t W, int32_t dtype, const PlanOpts &o,
                      Plan *p);
// Register bound of the backward's main kernel for width W.
inline int bwd_regs_bound(int64_t W) { return (W >= 4 && W <= kTwoCtaMaxW) ? kRegsTwoCta : kRegsOneCta; }

// CTA ranges of at least kDeepMinRowsPerCta rows stage every row with its own
// bulk copy, even where a stage's rows lie back to back in memory (B = 1, one
// H-block): many copies in flight beat one larger copy there. Shorter ranges
// (small problems) move adjacent rows with one copy per tensor.
inline bool long_ranges(const Plan &p) { return p.rows_total / p.ncta >= kDeepMinRowsPerCta; }

// First row of CTA c's range.
MCC1D_HD inline int64_t cta_row_begin(int64_t c, int64_t rows_total, int64_t ncta) {
    return c * rows_total / ncta;
}

}  // namespace mcc1d
