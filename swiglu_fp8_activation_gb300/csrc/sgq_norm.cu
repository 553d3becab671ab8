// sgq_norm.cu -- instantiations and launcher of the add + RMSNorm + quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using NormKernel = void (*)(const NormArgs);

template <int FMT, int LAYOUT, bool RES, bool FULL>
NormKernel pick(int nv) {
    switch (nv) {
        case 1: return norm_quant_kernel<FMT, LAYOUT, 1, RES, FULL>;
        case 2: return norm_quant_kernel<FMT, LAYOUT, 2, RES, FULL>;
        case 3: return norm_quant_kernel<FMT, LAYOUT, 3, RES, FULL>;
        default: return norm_quant_kernel<FMT, LAYOUT, 4, RES, FULL>;
    }
}

// The instantiated (format, scale layout) pairs: MX row-major or swizzled,
// 1x128 row- or column-major, per-token row-major.
template <bool RES, bool FULL>
NormKernel pick_fmt(int fmt, int layout, int nv) {
    if (fmt == FMT_MX)
        return layout == SCALE_SWIZZLED ? pick<FMT_MX, SCALE_SWIZZLED, RES, FULL>(nv)
                                        : pick<FMT_MX, SCALE_ROW_MAJOR, RES, FULL>(nv);
    if (fmt == FMT_B128)
        return layout == SCALE_COL_MAJOR ? pick<FMT_B128, SCALE_COL_MAJOR, RES, FULL>(nv)
                                         : pick<FMT_B128, SCALE_ROW_MAJOR, RES, FULL>(nv);
    return pick<FMT_PT, SCALE_ROW_MAJOR, RES, FULL>(nv);
}
}  // namespace

cudaError_t launch_norm(int fmt, const Plan& p, const NormArgs& a, cudaStream_t stream) {
    const int l = a.so.layout;
    NormKernel k = a.r_in ? (p.full ? pick_fmt<true, true>(fmt, l, p.nv) : pick_fmt<true, false>(fmt, l, p.nv))
                          : (p.full ? pick_fmt<false, true>(fmt, l, p.nv) : pick_fmt<false, false>(fmt, l, p.nv));
    return launch_pdl(k, p, a, stream, norm_stage_bytes(a.r_in != nullptr, p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
