// sgq_wide.cu -- instantiations and launchers of the kernels for rows wider
// than one CTA covers (kMaxTPR * kMaxNV * 8 columns): each row is split over
// the CTAs of a thread block cluster, which combine their partial sums of
// squares and amaxes through shared memory.
#include "sgq_launch.h"

namespace sgq {

namespace {
using NormKernel = void (*)(const NormArgs);

template <bool RES, int DT>
NormKernel pick_norm(int fmt, int layout) {
    if (fmt == FMT_MX)
        return layout == SCALE_SWIZZLED ? norm_cluster_kernel<FMT_MX, SCALE_SWIZZLED, RES, DT>
                                        : norm_cluster_kernel<FMT_MX, SCALE_ROW_MAJOR, RES, DT>;
    if (fmt == FMT_B128)
        return layout == SCALE_COL_MAJOR ? norm_cluster_kernel<FMT_B128, SCALE_COL_MAJOR, RES, DT>
                                         : norm_cluster_kernel<FMT_B128, SCALE_ROW_MAJOR, RES, DT>;
    return norm_cluster_kernel<FMT_PT, SCALE_ROW_MAJOR, RES, DT>;
}
}  // namespace

cudaError_t launch_norm_cluster(int fmt, int dt, const Plan& p, const NormArgs& a, cudaStream_t stream) {
    const int l = a.so.layout;
    const bool res = a.r_in != nullptr;
    NormKernel k = dt == DT_F16 ? (res ? pick_norm<true, DT_F16>(fmt, l) : pick_norm<false, DT_F16>(fmt, l))
                                : (res ? pick_norm<true, DT_BF16>(fmt, l) : pick_norm<false, DT_BF16>(fmt, l));
    return launch_pdl(k, p, a, stream, norm_stage_bytes(res, kMaxNV, p.tpr));
}

cudaError_t launch_swiglu_pt_cluster(const Plan& p, const SwigluArgs& a, bool clamp16, cudaStream_t stream) {
    void (*k)(const SwigluArgs) = a.act == ACT_SILU ? swiglu_pt_cluster_kernel<ACT_SILU, false>
                                  : clamp16         ? swiglu_pt_cluster_kernel<ACT_OAI, true>
                                                    : swiglu_pt_cluster_kernel<ACT_OAI, false>;
    return launch_pdl(k, p, a, stream, swiglu_stage_bytes(kMaxNV, p.tpr));
}

cudaError_t launch_quant_pt_cluster(int dt, const Plan& p, const QuantArgs& a, cudaStream_t stream) {
    void (*k)(const QuantArgs) = dt == DT_F16 ? quant_pt_cluster_kernel<DT_F16> : quant_pt_cluster_kernel<DT_BF16>;
    return launch_pdl(k, p, a, stream, quant_stage_bytes(kMaxNV, p.tpr));
}

}  // namespace sgq
