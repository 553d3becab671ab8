// sgq_swiglu.cu -- instantiations and launcher of the SwiGLU + quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using SwigluKernel = void (*)(const SwigluArgs);

template <int FMT, int LAYOUT, int ACT, bool FULL>
SwigluKernel pick(int nv) {
    switch (nv) {
        case 1: return swiglu_quant_kernel<FMT, LAYOUT, 1, ACT, FULL>;
        case 2: return swiglu_quant_kernel<FMT, LAYOUT, 2, ACT, FULL>;
        case 3: return swiglu_quant_kernel<FMT, LAYOUT, 3, ACT, FULL>;
        default: return swiglu_quant_kernel<FMT, LAYOUT, 4, ACT, FULL>;
    }
}

// The instantiated (format, scale layout) pairs, as for the norm.
template <int ACT, bool FULL>
SwigluKernel pick_fmt(int fmt, int layout, int nv) {
    if (fmt == FMT_MX)
        return layout == SCALE_SWIZZLED ? pick<FMT_MX, SCALE_SWIZZLED, ACT, FULL>(nv)
                                        : pick<FMT_MX, SCALE_ROW_MAJOR, ACT, FULL>(nv);
    if (fmt == FMT_B128)
        return layout == SCALE_COL_MAJOR ? pick<FMT_B128, SCALE_COL_MAJOR, ACT, FULL>(nv)
                                         : pick<FMT_B128, SCALE_ROW_MAJOR, ACT, FULL>(nv);
    return pick<FMT_PT, SCALE_ROW_MAJOR, ACT, FULL>(nv);
}
}  // namespace

cudaError_t launch_swiglu(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream) {
    const int l = a.so.layout;
    SwigluKernel k = a.act == ACT_OAI
                         ? (p.full ? pick_fmt<ACT_OAI, true>(fmt, l, p.nv) : pick_fmt<ACT_OAI, false>(fmt, l, p.nv))
                         : (p.full ? pick_fmt<ACT_SILU, true>(fmt, l, p.nv) : pick_fmt<ACT_SILU, false>(fmt, l, p.nv));
    return launch_pdl(k, p, a, stream, swiglu_stage_bytes(p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
