// sgq_dual.cu -- instantiations and launcher of the two-segment (q/kv) norm.
#include "sgq_launch.h"

namespace sgq {

namespace {
using DualKernel = void (*)(const DualArgs);

template <int FMT, int DT>
DualKernel pick(int nv) {
    switch (nv) {
        case 1: return norm_dual_kernel<FMT, 1, DT>;
        case 2: return norm_dual_kernel<FMT, 2, DT>;
        case 3: return norm_dual_kernel<FMT, 3, DT>;
        default: return norm_dual_kernel<FMT, 4, DT>;
    }
}

template <int DT>
DualKernel pick_fmt(int fmt, int nv) {
    return fmt == FMT_MX ? pick<FMT_MX, DT>(nv) : fmt == FMT_B128 ? pick<FMT_B128, DT>(nv) : pick<FMT_PT, DT>(nv);
}
}  // namespace

cudaError_t launch_norm_dual(int fmt, int dt, const Plan& p, const DualArgs& d, cudaStream_t stream) {
    DualKernel k = dt == DT_F16 ? pick_fmt<DT_F16>(fmt, p.nv) : pick_fmt<DT_BF16>(fmt, p.nv);
    return launch_pdl(k, p, d, stream, norm_stage_bytes(false, p.nv, p.rpc * p.tpr));
}

}  // namespace sgq
