// sgq_swiglu.cu -- instantiations and launcher of the SwiGLU + quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using SwigluKernel = void (*)(const SwigluArgs);

template <int FMT, int ACT>
SwigluKernel pick(int nv) {
    switch (nv) {
        case 1: return swiglu_quant_kernel<FMT, 1, ACT>;
        case 2: return swiglu_quant_kernel<FMT, 2, ACT>;
        case 3: return swiglu_quant_kernel<FMT, 3, ACT>;
        default: return swiglu_quant_kernel<FMT, 4, ACT>;
    }
}

template <int ACT>
SwigluKernel pick_fmt(int fmt, int nv) {
    return fmt == FMT_MX ? pick<FMT_MX, ACT>(nv) : fmt == FMT_B128 ? pick<FMT_B128, ACT>(nv) : pick<FMT_PT, ACT>(nv);
}
}  // namespace

cudaError_t launch_swiglu(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream) {
    SwigluKernel k = a.act == ACT_OAI ? pick_fmt<ACT_OAI>(fmt, p.nv) : pick_fmt<ACT_SILU>(fmt, p.nv);
    return launch_pdl(k, p, a, stream, swiglu_stage_bytes(p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
