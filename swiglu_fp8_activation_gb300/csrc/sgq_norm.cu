// sgq_norm.cu -- instantiations and launcher of the add + RMSNorm + quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using NormKernel = void (*)(const NormArgs);

template <int FMT, bool RES>
NormKernel pick(int nv) {
    switch (nv) {
        case 1: return norm_quant_kernel<FMT, 1, RES>;
        case 2: return norm_quant_kernel<FMT, 2, RES>;
        case 3: return norm_quant_kernel<FMT, 3, RES>;
        default: return norm_quant_kernel<FMT, 4, RES>;
    }
}

template <bool RES>
NormKernel pick_fmt(int fmt, int nv) {
    return fmt == FMT_MX ? pick<FMT_MX, RES>(nv) : fmt == FMT_B128 ? pick<FMT_B128, RES>(nv) : pick<FMT_PT, RES>(nv);
}
}  // namespace

cudaError_t launch_norm(int fmt, const Plan& p, const NormArgs& a, cudaStream_t stream) {
    NormKernel k = a.r_in ? pick_fmt<true>(fmt, p.nv) : pick_fmt<false>(fmt, p.nv);
    return launch_pdl(k, p, a, stream, norm_stage_bytes(a.r_in != nullptr, p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
