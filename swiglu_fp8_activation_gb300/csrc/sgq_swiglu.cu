// sgq_swiglu.cu -- the SwiGLU + quant kernel for the OAI activation, and the
// launcher that picks the activation.
#include "sgq_swiglu_impl.cuh"

namespace sgq {

cudaError_t launch_swiglu(int fmt, const Plan& p, const SwigluArgs& a, bool clamp16, cudaStream_t stream) {
    if (a.act != ACT_OAI) return launch_swiglu_silu(fmt, p, a, stream);
    return clamp16 ? SwigluPick<ACT_OAI, true>::launch(fmt, p, a, stream)
                   : SwigluPick<ACT_OAI, false>::launch(fmt, p, a, stream);
}

}  // namespace sgq
