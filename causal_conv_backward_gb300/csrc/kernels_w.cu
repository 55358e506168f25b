// kernels_w.cu - instances of the backward's main kernel for widths W other
// than 3 (one rows-per-stage choice, R = 6; R = 8 at W = 8), for the strided entry points,
// which accept 1 <= W <= 8. Widths from 4 up keep 4 channels per thread so
// their W accumulators per channel stay in registers; widths 4 and 5 run two
// CTAs per SM under the matching register bound. Compiled apart from
// kernels.cu so the two build in parallel.
#include "bwd_main.cuh"

namespace mcc1d {

template <int DT, int W>
static MainFn pick(int vec, int R)
{
    if constexpr (W == kMaxW)
        return vec == 4 && R == 8 ? mcc1d_bwd_main<DT, 8, 2, W> : nullptr;
    else if constexpr (W >= 4 && W <= kTwoCtaMaxW)
        return vec == 4 && R == 6 ? mcc1d_bwd_main_x2<DT, 6, 2, W> : nullptr;
    else if constexpr (W >= 4)
        return vec == 4 && R == 6 ? mcc1d_bwd_main<DT, 6, 2, W> : nullptr;
    else if (R == 6)
        return vec == 4 ? mcc1d_bwd_main<DT, 6, 2, W> : mcc1d_bwd_main<DT, 6, 4, W>;
    return nullptr;
}

template <int DT>
static MainFn pick_w(int vec, int W, int R)
{
    switch (W) {
    case 1: return pick<DT, 1>(vec, R);
    case 2: return pick<DT, 2>(vec, R);
    case 4: return pick<DT, 4>(vec, R);
    case 5: return pick<DT, 5>(vec, R);
    case 6: return pick<DT, 6>(vec, R);
    case 7: return pick<DT, 7>(vec, R);
    case 8: return pick<DT, 8>(vec, R);
    default: return nullptr;
    }
}

MainFn main_kernel_other_w(int dtype, int vec, int W, int R)
{
    return dtype == 0 ? pick_w<0>(vec, W, R) : pick_w<1>(vec, W, R);
}

}  // namespace mcc1d
