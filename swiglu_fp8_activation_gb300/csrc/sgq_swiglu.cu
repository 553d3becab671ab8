// sgq_swiglu.cu -- the exact-fit SwiGLU + quant kernels for the OAI
// activation, and the launcher that picks the activation and the kernel set.
#include "sgq_swiglu_impl.cuh"

namespace sgq {

cudaError_t launch_swiglu_oai_full(int fmt, const Plan& p, const SwigluArgs& a, bool clamp16, cudaStream_t stream) {
    return clamp16 ? SwigluPick<ACT_OAI, true>::launch<true>(fmt, p, a, stream)
                   : SwigluPick<ACT_OAI, false>::launch<true>(fmt, p, a, stream);
}

cudaError_t launch_swiglu(int fmt, const Plan& p, const SwigluArgs& a, bool clamp16, cudaStream_t stream) {
    if (a.act != ACT_OAI)
        return p.full ? launch_swiglu_silu_full(fmt, p, a, stream) : launch_swiglu_silu_part(fmt, p, a, stream);
    return p.full ? launch_swiglu_oai_full(fmt, p, a, clamp16, stream)
                  : launch_swiglu_oai_part(fmt, p, a, clamp16, stream);
}

}  // namespace sgq
