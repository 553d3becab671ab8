// sgq_swiglu_silu.cu -- the exact-fit SwiGLU + quant kernels for SiLU-and-mul.
#include "sgq_swiglu_impl.cuh"

namespace sgq {

cudaError_t launch_swiglu_silu_full(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream) {
    return SwigluPick<ACT_SILU, false>::launch<true>(fmt, p, a, stream);
}

}  // namespace sgq
