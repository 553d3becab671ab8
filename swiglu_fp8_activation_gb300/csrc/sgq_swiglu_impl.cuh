// sgq_swiglu_impl.cuh -- kernel selection and launch of the SwiGLU + quant
// kernel; included by the translation units that instantiate it (OAI and
// SiLU-and-mul, each exact-fit and bounds-checked), which compile in
// parallel.
#pragma once

#include "sgq_launch.h"

namespace sgq {
namespace {

template <int ACT, bool CLAMP16>
struct SwigluPick {
    using Kernel = void (*)(const SwigluArgs);

    // SiLU-and-mul in the MX and 1x128 formats takes the register-capped kernels.
    template <int FMT, int LAYOUT, int NV, bool FULL>
    static Kernel kernel() {
        if constexpr (ACT == ACT_SILU && FMT != FMT_PT)
            return swiglu_quant_kernel_r56<FMT, LAYOUT, NV, ACT, FULL, CLAMP16>;
        else
            return swiglu_quant_kernel<FMT, LAYOUT, NV, ACT, FULL, CLAMP16>;
    }

    template <int FMT, int LAYOUT, bool FULL>
    static Kernel pick(int nv) {
        switch (nv) {
            case 1: return kernel<FMT, LAYOUT, 1, FULL>();
            case 2: return kernel<FMT, LAYOUT, 2, FULL>();
            case 3: return kernel<FMT, LAYOUT, 3, FULL>();
            default: return kernel<FMT, LAYOUT, 4, FULL>();
        }
    }

    // The instantiated (format, scale layout) pairs, as for the norm.
    template <bool FULL>
    static Kernel pick_fmt(int fmt, int layout, int nv) {
        if (fmt == FMT_MX)
            return layout == SCALE_SWIZZLED ? pick<FMT_MX, SCALE_SWIZZLED, FULL>(nv)
                                            : pick<FMT_MX, SCALE_ROW_MAJOR, FULL>(nv);
        if (fmt == FMT_B128)
            return layout == SCALE_COL_MAJOR ? pick<FMT_B128, SCALE_COL_MAJOR, FULL>(nv)
                                             : pick<FMT_B128, SCALE_ROW_MAJOR, FULL>(nv);
        return pick<FMT_PT, SCALE_ROW_MAJOR, FULL>(nv);
    }

    // The exact-fit (FULL) and the bounds-checked kernels are instantiated in
    // separate translation units, which compile in parallel.
    template <bool FULL>
    static cudaError_t launch(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream) {
        Kernel k = pick_fmt<FULL>(fmt, a.so.layout, p.nv);
        return launch_pdl(k, p, a, stream, swiglu_stage_bytes(p.nv, p.rpc * p.tpr));
    }
};

}  // namespace
}  // namespace sgq
