// sgq_swiglu_part.cu -- the bounds-checked SwiGLU + quant kernels for the
// OAI activation.
#include "sgq_swiglu_impl.cuh"

namespace sgq {

cudaError_t launch_swiglu_oai_part(int fmt, const Plan& p, const SwigluArgs& a, bool clamp16, cudaStream_t stream) {
    return clamp16 ? SwigluPick<ACT_OAI, true>::launch<false>(fmt, p, a, stream)
                   : SwigluPick<ACT_OAI, false>::launch<false>(fmt, p, a, stream);
}

}  // namespace sgq
