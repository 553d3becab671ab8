// sgq_swiglu.cu -- instantiations and launcher of the SwiGLU + quant kernel.
#include "sgq_launch.h"

namespace sgq {

namespace {
using SwigluKernel = void (*)(const SwigluArgs);

template <int FMT>
SwigluKernel pick(int nv) {
    switch (nv) {
        case 1: return swiglu_quant_kernel<FMT, 1>;
        case 2: return swiglu_quant_kernel<FMT, 2>;
        case 3: return swiglu_quant_kernel<FMT, 3>;
        default: return swiglu_quant_kernel<FMT, 4>;
    }
}
}  // namespace

cudaError_t launch_swiglu(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream) {
    SwigluKernel k = fmt == FMT_MX ? pick<FMT_MX>(p.nv) : fmt == FMT_B128 ? pick<FMT_B128>(p.nv) : pick<FMT_PT>(p.nv);
    k<<<(unsigned)p.grid, (unsigned)(p.rpc * p.tpr), 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sgq
