// sgq_allreduce.cu -- instantiations and launcher of the norm with the
// tensor-parallel all-reduce folded in (x = the ranks' partial rows summed).
#include "sgq_launch.h"

namespace sgq {

namespace {
using NormKernel = void (*)(const NormARArgs);

template <int FMT, int LAYOUT, bool RES, bool FULL>
NormKernel pick_nv(int nv) {
    switch (nv) {
        case 1: return norm_ar_kernel<FMT, LAYOUT, 1, RES, FULL>;
        case 2: return norm_ar_kernel<FMT, LAYOUT, 2, RES, FULL>;
        case 3: return norm_ar_kernel<FMT, LAYOUT, 3, RES, FULL>;
        default: return norm_ar_kernel<FMT, LAYOUT, 4, RES, FULL>;
    }
}

template <bool RES, bool FULL>
NormKernel pick_fmt(int fmt, int layout, int nv) {
    if (fmt == FMT_MX)
        return layout == SCALE_SWIZZLED ? pick_nv<FMT_MX, SCALE_SWIZZLED, RES, FULL>(nv)
                                        : pick_nv<FMT_MX, SCALE_ROW_MAJOR, RES, FULL>(nv);
    if (fmt == FMT_B128)
        return layout == SCALE_COL_MAJOR ? pick_nv<FMT_B128, SCALE_COL_MAJOR, RES, FULL>(nv)
                                         : pick_nv<FMT_B128, SCALE_ROW_MAJOR, RES, FULL>(nv);
    return pick_nv<FMT_PT, SCALE_ROW_MAJOR, RES, FULL>(nv);
}
}  // namespace

cudaError_t launch_norm_ar(int fmt, const Plan& p, const NormARArgs& aa, cudaStream_t stream) {
    const int l = aa.a.so.layout;
    const bool res = aa.a.r_in != nullptr;
    NormKernel k = res ? (p.full ? pick_fmt<true, true>(fmt, l, p.nv) : pick_fmt<true, false>(fmt, l, p.nv))
                       : (p.full ? pick_fmt<false, true>(fmt, l, p.nv) : pick_fmt<false, false>(fmt, l, p.nv));
    return launch_pdl(k, p, aa, stream, norm_ar_stage_bytes(res, aa.ar.n, p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
