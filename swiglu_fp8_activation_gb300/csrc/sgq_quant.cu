// sgq_quant.cu -- instantiations and launcher of the standalone quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using QuantKernel = void (*)(const QuantArgs);

template <int FMT, bool FULL>
QuantKernel pick(int nv) {
    switch (nv) {
        case 1: return quant_kernel<FMT, 1, FULL>;
        case 2: return quant_kernel<FMT, 2, FULL>;
        case 3: return quant_kernel<FMT, 3, FULL>;
        default: return quant_kernel<FMT, 4, FULL>;
    }
}

template <bool FULL>
QuantKernel pick_fmt(int fmt, int nv) {
    return fmt == FMT_MX ? pick<FMT_MX, FULL>(nv) : fmt == FMT_B128 ? pick<FMT_B128, FULL>(nv) : pick<FMT_PT, FULL>(nv);
}
}  // namespace

cudaError_t launch_quant(int fmt, const Plan& p, const QuantArgs& a, cudaStream_t stream) {
    QuantKernel k = p.full ? pick_fmt<true>(fmt, p.nv) : pick_fmt<false>(fmt, p.nv);
    return launch_pdl(k, p, a, stream, quant_stage_bytes(p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
