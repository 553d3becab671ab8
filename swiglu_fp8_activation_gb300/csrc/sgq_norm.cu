// sgq_norm.cu -- the add + RMSNorm + quant kernel on bf16 activations, and
// the launcher that picks the activation type.
#include "sgq_norm_impl.cuh"

namespace sgq {

cudaError_t launch_norm(int fmt, int dt, const Plan& p, const NormArgs& a, cudaStream_t stream) {
    if (dt == DT_F16) return launch_norm_f16(fmt, p, a, stream);
    return NormPick<DT_BF16>::launch(fmt, p, a, stream);
}

cudaError_t launch_norm_pt_persistent(int dt, const Plan& p, const NormArgs& a, cudaStream_t stream) {
    if (dt == DT_F16) return launch_norm_pt_persistent_f16(p, a, stream);
    return NormPick<DT_BF16>::launch_persistent(p, a, stream);
}

}  // namespace sgq
