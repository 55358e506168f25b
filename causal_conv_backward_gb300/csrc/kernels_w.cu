// kernels_w.cu - instances of the backward's main kernel for widths W other
// than 3 (one rows-per-stage choice, R = 6), for the strided entry points,
// which accept 1 <= W <= 8. Widths from 4 up keep 4 channels per thread so
// their W accumulators per channel stay in registers; widths 4 and 5 run two
// CTAs per SM under the matching register bound. Compiled apart from
// kernels.cu so the two build in parallel.
#include "bwd_main.cuh"

namespace mcc1d {

template <int DT, int W>
static MainFn pick(int vec)
{
    if constexpr (W >= 4 && W <= kTwoCtaMaxW)
        return vec == 4 ? mcc1d_bwd_main_x2<DT, 6, 2, W> : nullptr;
    else if constexpr (W >= 4)
        return vec == 4 ? mcc1d_bwd_main<DT, 6, 2, W> : nullptr;
    else
        return vec == 4 ? mcc1d_bwd_main<DT, 6, 2, W> : mcc1d_bwd_main<DT, 6, 4, W>;
}

template <int DT>
static MainFn pick_w(int vec, int W)
{
    switch (W) {
    case 1: return pick<DT, 1>(vec);
    case 2: return pick<DT, 2>(vec);
    case 4: return pick<DT, 4>(vec);
    case 5: return pick<DT, 5>(vec);
    case 6: return pick<DT, 6>(vec);
    case 7: return pick<DT, 7>(vec);
    case 8: return pick<DT, 8>(vec);
    default: return nullptr;
    }
}

MainFn main_kernel_other_w(int dtype, int vec, int W)
{
    return dtype == 0 ? pick_w<0>(vec, W) : pick_w<1>(vec, W);
}

}  // namespace mcc1d
