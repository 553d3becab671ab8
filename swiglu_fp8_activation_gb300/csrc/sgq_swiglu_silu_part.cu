// sgq_swiglu_silu_part.cu -- the bounds-checked SwiGLU + quant kernels for
// SiLU-and-mul.
#include "sgq_swiglu_impl.cuh"

namespace sgq {

cudaError_t launch_swiglu_silu_part(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream) {
    return SwigluPick<ACT_SILU, false>::launch<false>(fmt, p, a, stream);
}

}  // namespace sgq
