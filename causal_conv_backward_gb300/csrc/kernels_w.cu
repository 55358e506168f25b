// kernels_w.cu - instances of the backward's main kernel for widths W other
// than 3 (one rows-per-stage choice: R = 6; 10 at W = 4..6, 8 at W = 7, 8), for
// the strided entry points, which accept 1 <= W <= 8. Widths from 4 up keep 4 channels
// per thread so their W accumulators per channel stay in registers; width 4
// runs two CTAs per SM under the matching register bound; widths from 5
// split the register file by warpgroup when an H-block needs more than one
// consumer warpgroup (mcc1d_bwd_main_rs), else run the plain one-CTA form.
// Compiled apart from kernels.cu so the two build in parallel.
#include "bwd_main.cuh"

namespace mcc1d {

template <int DT, int W>
static MainFn pick(int vec, int R, bool split)
{
    constexpr int kR = W >= 4 && W <= 6 ? 10 : W >= 7 ? 8 : 6;   // as the plan's rows per stage
    if (R != kR)
        return nullptr;
    if constexpr (W >= kSplitMinW) {
        if (vec != 4)
            return nullptr;
        return split ? mcc1d_bwd_main_rs<DT, kR, 2, W> : mcc1d_bwd_main<DT, kR, 2, W>;
    } else {
        if (split)
            return nullptr;
        if constexpr (W >= 4 && W <= kTwoCtaMaxW)
            return vec == 4 ? mcc1d_bwd_main_x2<DT, kR, 2, W> : nullptr;
        else if constexpr (W >= 4)
            return vec == 4 ? mcc1d_bwd_main<DT, kR, 2, W> : nullptr;
        else
            return vec == 4 ? mcc1d_bwd_main<DT, kR, 2, W> : mcc1d_bwd_main<DT, kR, 4, W>;
    }
}

template <int DT>
static MainFn pick_w(int vec, int W, int R, bool split)
{
    switch (W) {
    case 1: return pick<DT, 1>(vec, R, split);
    case 2: return pick<DT, 2>(vec, R, split);
    case 4: return pick<DT, 4>(vec, R, split);
    case 5: return pick<DT, 5>(vec, R, split);
    case 6: return pick<DT, 6>(vec, R, split);
    case 7: return pick<DT, 7>(vec, R, split);
    case 8: return pick<DT, 8>(vec, R, split);
    default: return nullptr;
    }
}

MainFn main_kernel_other_w(int dtype, int vec, int W, int R, bool split)
{
    return dtype == 0 ? pick_w<0>(vec, W, R, split) : pick_w<1>(vec, W, R, split);
}

}  // namespace mcc1d
