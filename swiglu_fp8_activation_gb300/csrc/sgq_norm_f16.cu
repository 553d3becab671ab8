// sgq_norm_f16.cu -- the add + RMSNorm + quant kernel on fp16 activations.
#include "sgq_norm_impl.cuh"

namespace sgq {

cudaError_t launch_norm_f16(int fmt, const Plan& p, const NormArgs& a, cudaStream_t stream) {
    return NormPick<DT_F16>::launch(fmt, p, a, stream);
}

cudaError_t launch_norm_pt_persistent_f16(const Plan& p, const NormArgs& a, cudaStream_t stream) {
    return NormPick<DT_F16>::launch_persistent(p, a, stream);
}

}  // namespace sgq
