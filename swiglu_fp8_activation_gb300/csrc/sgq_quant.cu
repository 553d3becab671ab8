// sgq_quant.cu -- instantiations and launcher of the standalone quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using QuantKernel = void (*)(const QuantArgs);

template <int FMT, int LAYOUT, bool FULL, int DT>
QuantKernel pick(int nv) {
    switch (nv) {
        case 1: return quant_kernel<FMT, LAYOUT, 1, FULL, DT>;
        case 2: return quant_kernel<FMT, LAYOUT, 2, FULL, DT>;
        case 3: return quant_kernel<FMT, LAYOUT, 3, FULL, DT>;
        default: return quant_kernel<FMT, LAYOUT, 4, FULL, DT>;
    }
}

// The instantiated (format, scale layout) pairs, as for the norm.
template <bool FULL, int DT>
QuantKernel pick_fmt(int fmt, int layout, int nv) {
    if (fmt == FMT_MX)
        return layout == SCALE_SWIZZLED ? pick<FMT_MX, SCALE_SWIZZLED, FULL, DT>(nv)
                                        : pick<FMT_MX, SCALE_ROW_MAJOR, FULL, DT>(nv);
    if (fmt == FMT_B128)
        return layout == SCALE_COL_MAJOR ? pick<FMT_B128, SCALE_COL_MAJOR, FULL, DT>(nv)
                                         : pick<FMT_B128, SCALE_ROW_MAJOR, FULL, DT>(nv);
    return pick<FMT_PT, SCALE_ROW_MAJOR, FULL, DT>(nv);
}
}  // namespace

cudaError_t launch_quant(int fmt, int dt, const Plan& p, const QuantArgs& a, cudaStream_t stream) {
    const int l = a.so.layout;
    QuantKernel k = dt == DT_F16 ? (p.full ? pick_fmt<true, DT_F16>(fmt, l, p.nv) : pick_fmt<false, DT_F16>(fmt, l, p.nv))
                                 : (p.full ? pick_fmt<true, DT_BF16>(fmt, l, p.nv) : pick_fmt<false, DT_BF16>(fmt, l, p.nv));
    return launch_pdl(k, p, a, stream, quant_stage_bytes(p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
