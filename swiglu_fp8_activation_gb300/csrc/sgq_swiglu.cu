// sgq_swiglu.cu -- instantiations and launcher of the SwiGLU + quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using SwigluKernel = void (*)(const SwigluArgs);

template <int FMT, int ACT, bool FULL>
SwigluKernel pick(int nv) {
    switch (nv) {
        case 1: return swiglu_quant_kernel<FMT, 1, ACT, FULL>;
        case 2: return swiglu_quant_kernel<FMT, 2, ACT, FULL>;
        case 3: return swiglu_quant_kernel<FMT, 3, ACT, FULL>;
        default: return swiglu_quant_kernel<FMT, 4, ACT, FULL>;
    }
}

template <int ACT, bool FULL>
SwigluKernel pick_fmt(int fmt, int nv) {
    return fmt == FMT_MX ? pick<FMT_MX, ACT, FULL>(nv)
                         : fmt == FMT_B128 ? pick<FMT_B128, ACT, FULL>(nv) : pick<FMT_PT, ACT, FULL>(nv);
}
}  // namespace

cudaError_t launch_swiglu(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream) {
    SwigluKernel k = a.act == ACT_OAI ? (p.full ? pick_fmt<ACT_OAI, true>(fmt, p.nv) : pick_fmt<ACT_OAI, false>(fmt, p.nv))
                                      : (p.full ? pick_fmt<ACT_SILU, true>(fmt, p.nv) : pick_fmt<ACT_SILU, false>(fmt, p.nv));
    return launch_pdl(k, p, a, stream, swiglu_stage_bytes(p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
