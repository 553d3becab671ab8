// sgq_norm.cu -- instantiations and launcher of the add + RMSNorm + quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using NormKernel = void (*)(const NormArgs);

template <int FMT, bool RES, bool FULL>
NormKernel pick(int nv) {
    switch (nv) {
        case 1: return norm_quant_kernel<FMT, 1, RES, FULL>;
        case 2: return norm_quant_kernel<FMT, 2, RES, FULL>;
        case 3: return norm_quant_kernel<FMT, 3, RES, FULL>;
        default: return norm_quant_kernel<FMT, 4, RES, FULL>;
    }
}

template <bool RES, bool FULL>
NormKernel pick_fmt(int fmt, int nv) {
    return fmt == FMT_MX ? pick<FMT_MX, RES, FULL>(nv)
                         : fmt == FMT_B128 ? pick<FMT_B128, RES, FULL>(nv) : pick<FMT_PT, RES, FULL>(nv);
}
}  // namespace

cudaError_t launch_norm(int fmt, const Plan& p, const NormArgs& a, cudaStream_t stream) {
    NormKernel k = a.r_in ? (p.full ? pick_fmt<true, true>(fmt, p.nv) : pick_fmt<true, false>(fmt, p.nv))
                          : (p.full ? pick_fmt<false, true>(fmt, p.nv) : pick_fmt<false, false>(fmt, p.nv));
    return launch_pdl(k, p, a, stream, norm_stage_bytes(a.r_in != nullptr, p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
