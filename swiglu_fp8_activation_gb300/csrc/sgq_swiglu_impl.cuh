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

    // SiLU-and-mul in the MX and 1x128 formats has register-capped kernels
    // too, taken (r56) when the grid is larger than one wave of the uncapped
    // kernels (two CTAs an SM): there the extra resident CTA pays (11% at
    // M = 2048, I = 12288), within one wave the uncapped kernels are faster
    // (5.3 against 6.7 us at M = 256).
    static constexpr bool kHasR56 = ACT == ACT_SILU;

    template <int FMT, int LAYOUT, int NV, bool FULL>
    static Kernel kernel(bool r56) {
        if constexpr (kHasR56 && FMT != FMT_PT) {
            if (r56) return swiglu_quant_kernel_r56<FMT, LAYOUT, NV, ACT, FULL, CLAMP16>;
        }
        return swiglu_quant_kernel<FMT, LAYOUT, NV, ACT, FULL, CLAMP16>;
    }

    template <int FMT, int LAYOUT, bool FULL>
    static Kernel pick(int nv, bool r56) {
        switch (nv) {
            case 1: return kernel<FMT, LAYOUT, 1, FULL>(r56);
            case 2: return kernel<FMT, LAYOUT, 2, FULL>(r56);
            case 3: return kernel<FMT, LAYOUT, 3, FULL>(r56);
            default: return kernel<FMT, LAYOUT, 4, FULL>(r56);
        }
    }

    // The instantiated (format, scale layout) pairs, as for the norm.
    template <bool FULL>
    static Kernel pick_fmt(int fmt, int layout, int nv, bool r56) {
        if (fmt == FMT_MX)
            return layout == SCALE_SWIZZLED ? pick<FMT_MX, SCALE_SWIZZLED, FULL>(nv, r56)
                                            : pick<FMT_MX, SCALE_ROW_MAJOR, FULL>(nv, r56);
        if (fmt == FMT_B128)
            return layout == SCALE_COL_MAJOR ? pick<FMT_B128, SCALE_COL_MAJOR, FULL>(nv, r56)
                                             : pick<FMT_B128, SCALE_ROW_MAJOR, FULL>(nv, r56);
        return pick<FMT_PT, SCALE_ROW_MAJOR, FULL>(nv, r56);
    }

    // The exact-fit (FULL) and the bounds-checked kernels are instantiated in
    // separate translation units, which compile in parallel.
    template <bool FULL>
    static cudaError_t launch(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream) {
        const bool r56 = kHasR56 && p.sms > 0 && p.grid > 2 * (int64_t)p.sms;
        Kernel k = pick_fmt<FULL>(fmt, a.so.layout, p.nv, r56);
        return launch_pdl(k, p, a, stream, swiglu_stage_bytes(p.nv, p.rpc * p.tpr));
    }
};

}  // namespace
}  // namespace sgq
