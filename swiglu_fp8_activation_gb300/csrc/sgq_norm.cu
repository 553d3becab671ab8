// sgq_norm.cu -- instantiations and launcher of the add + RMSNorm + quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using NormKernel = void (*)(const NormArgs);

template <int FMT>
NormKernel pick(int nv) {
    switch (nv) {
        case 1: return norm_quant_kernel<FMT, 1>;
        case 2: return norm_quant_kernel<FMT, 2>;
        case 3: return norm_quant_kernel<FMT, 3>;
        default: return norm_quant_kernel<FMT, 4>;
    }
}
}  // namespace

cudaError_t launch_norm(int fmt, const Plan& p, const NormArgs& a, cudaStream_t stream) {
    NormKernel k = fmt == FMT_MX ? pick<FMT_MX>(p.nv) : fmt == FMT_B128 ? pick<FMT_B128>(p.nv) : pick<FMT_PT>(p.nv);
    return launch_pdl(k, p, a, stream);
}

}  // namespace sgq
