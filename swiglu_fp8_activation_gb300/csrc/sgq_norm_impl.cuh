// sgq_norm_impl.cuh -- kernel selection and launch of the add + RMSNorm +
// quant kernel for one 16-bit activation type; included by the two
// translation units that instantiate it (bf16 and fp16), which compile in
// parallel.
#pragma once

#include "sgq_launch.h"

namespace sgq {
namespace {

template <int DT>
struct NormPick {
    using Kernel = void (*)(const NormArgs);

    template <int FMT, int LAYOUT, bool RES, bool FULL>
    static Kernel pick(int nv) {
        switch (nv) {
            case 1: return norm_quant_kernel<FMT, LAYOUT, 1, RES, FULL, DT>;
            case 2: return norm_quant_kernel<FMT, LAYOUT, 2, RES, FULL, DT>;
            case 3: return norm_quant_kernel<FMT, LAYOUT, 3, RES, FULL, DT>;
            default: return norm_quant_kernel<FMT, LAYOUT, 4, RES, FULL, DT>;
        }
    }

    // The instantiated (format, scale layout) pairs: MX row-major or
    // swizzled, 1x128 row- or column-major, per-token row-major.
    template <bool RES, bool FULL>
    static Kernel pick_fmt(int fmt, int layout, int nv) {
        if (fmt == FMT_MX)
            return layout == SCALE_SWIZZLED ? pick<FMT_MX, SCALE_SWIZZLED, RES, FULL>(nv)
                                            : pick<FMT_MX, SCALE_ROW_MAJOR, RES, FULL>(nv);
        if (fmt == FMT_B128)
            return layout == SCALE_COL_MAJOR ? pick<FMT_B128, SCALE_COL_MAJOR, RES, FULL>(nv)
                                             : pick<FMT_B128, SCALE_ROW_MAJOR, RES, FULL>(nv);
        return pick<FMT_PT, SCALE_ROW_MAJOR, RES, FULL>(nv);
    }

    static Kernel pick_persistent(int nv) {
        switch (nv) {
            case 1: return norm_pt_persistent_kernel<1, DT>;
            case 2: return norm_pt_persistent_kernel<2, DT>;
            case 3: return norm_pt_persistent_kernel<3, DT>;
            default: return norm_pt_persistent_kernel<4, DT>;
        }
    }

    // The persistent per-token norm: as many CTAs as fit on the device at
    // once (at most one per row block).
    static cudaError_t launch_persistent(const Plan& p, const NormArgs& a, cudaStream_t stream) {
        Kernel k = pick_persistent(p.nv);
        const int threads = p.rpc * p.tpr;
        const int smem = norm_pt_persistent_bytes(p.nv, threads);
        int per_sm = 0;
        const cudaError_t e = ctas_per_sm(reinterpret_cast<const void*>(k), p.device, threads, smem, &per_sm);
        if (e != cudaSuccess) return e;
        Plan q = p;
        const int64_t nblk = a.M / p.rpc, wave = (int64_t)(per_sm > 0 ? per_sm : 1) * p.sms;
        q.grid = nblk < wave ? nblk : wave;
        return launch_pdl(k, q, a, stream, smem);
    }

    static cudaError_t launch(int fmt, const Plan& p, const NormArgs& a, cudaStream_t stream) {
        const int l = a.so.layout;
        Kernel k = a.r_in ? (p.full ? pick_fmt<true, true>(fmt, l, p.nv) : pick_fmt<true, false>(fmt, l, p.nv))
                          : (p.full ? pick_fmt<false, true>(fmt, l, p.nv) : pick_fmt<false, false>(fmt, l, p.nv));
        return launch_pdl(k, p, a, stream, norm_stage_bytes(a.r_in != nullptr, p.nv, p.rpc * p.tpr));
    }
};

}  // namespace
}  // namespace sgq
