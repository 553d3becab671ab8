// sgq_quant.cu -- instantiations and launcher of the standalone quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using QuantKernel = void (*)(const QuantArgs);

template <int FMT, int LAYOUT, bool FULL>
QuantKernel pick(int nv) {
    switch (nv) {
        case 1: return quant_kernel<FMT, LAYOUT, 1, FULL>;
        case 2: return quant_kernel<FMT, LAYOUT, 2, FULL>;
        case 3: return quant_kernel<FMT, LAYOUT, 3, FULL>;
        default: return quant_kernel<FMT, LAYOUT, 4, FULL>;
    }
}

// The instantiated (format, scale layout) pairs, as for the norm.
template <bool FULL>
QuantKernel pick_fmt(int fmt, int layout, int nv) {
    if (fmt == FMT_MX)
        return layout == SCALE_SWIZZLED ? pick<FMT_MX, SCALE_SWIZZLED, FULL>(nv) : pick<FMT_MX, SCALE_ROW_MAJOR, FULL>(nv);
    if (fmt == FMT_B128)
        return layout == SCALE_COL_MAJOR ? pick<FMT_B128, SCALE_COL_MAJOR, FULL>(nv)
                                         : pick<FMT_B128, SCALE_ROW_MAJOR, FULL>(nv);
    return pick<FMT_PT, SCALE_ROW_MAJOR, FULL>(nv);
}
}  // namespace

cudaError_t launch_quant(int fmt, const Plan& p, const QuantArgs& a, cudaStream_t stream) {
    QuantKernel k = p.full ? pick_fmt<true>(fmt, a.so.layout, p.nv) : pick_fmt<false>(fmt, a.so.layout, p.nv);
    return launch_pdl(k, p, a, stream, quant_stage_bytes(p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
