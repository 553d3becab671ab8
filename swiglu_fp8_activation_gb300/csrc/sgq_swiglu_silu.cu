// sgq_swiglu_silu.cu -- the SwiGLU + quant kernel for SiLU-and-mul.
#include "sgq_swiglu_impl.cuh"

namespace sgq {

cudaError_t launch_swiglu_silu(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream) {
    return SwigluPick<ACT_SILU, false>::launch(fmt, p, a, stream);
}

}  // namespace sgq
