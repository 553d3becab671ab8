// sgq_launch.h -- host-side launchers of the row-engine kernels (one
// translation unit per operation, so they compile in parallel).
#pragma once

#include <cuda_runtime.h>

#include "sgq_kernels.cuh"

namespace sgq {

// Launch geometry of one call: `nv` chunks per thread, `tpr` threads per row,
// `rpc` rows per CTA, `grid` CTAs (times `seg` column segments a row, the
// grid's second dimension, for the launches that split rows).
struct Plan {
    int nv;
    int tpr;
    int rpc;
    int64_t grid;
    bool full;   // W/8 == tpr * nv and M % rpc == 0: no bounds checks needed
    int sms;     // multiprocessors of the device (0 if unknown)
    int seg = 1;
    int device = -1;   // the current device, for the per-device kernel attributes
    int cluster = 0;   // > 1: CTAs a thread block cluster (the grid is rows x cluster CTAs, one row each)
};

// Pick a plan for M rows of width W (W % 8 == 0). Returns false when W needs
// more than kMaxTPR threads per row.
bool plan_rows(int64_t M, int W, int sm_count, Plan* p);

// Kernels above 48 KB of static plus dynamic shared memory must opt in once
// per device; the library records the largest opt-in given to each kernel on
// each device, so that a launch calls cudaFuncSetAttribute only the first time
// it needs more than was granted before (a mutex-guarded table lookup else).
cudaError_t ensure_dynamic_smem(const void* kernel, int device, int bytes);

// CTAs of `threads` threads and `smem` bytes of dynamic shared memory that
// fit on one multiprocessor at once (the occupancy calculator's answer,
// recorded per kernel, device and shape, so that it is asked once).
cudaError_t ctas_per_sm(const void* kernel, int device, int threads, int smem, int* out);

// Launch kernel k on `stream` with programmatic stream serialisation: the
// grid may begin launching while the preceding kernel on the stream finishes
// (the kernels wait in pdl_wait() before touching memory the preceding grid
// may write). The result is cudaLaunchKernelEx's own, which reports the
// configuration and launch errors of this launch; a sticky or pending error
// left on the thread by unrelated work is neither read nor cleared.
template <typename Args>
cudaError_t launch_pdl(void (*k)(const Args), const Plan& p, const Args& a, cudaStream_t stream,
                       int dynamic_smem = 0) {
    // (static shared memory here is a few hundred bytes)
    if (dynamic_smem > 40 * 1024) {
        const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(k), p.device, dynamic_smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid, (unsigned)p.seg);
    cfg.blockDim = dim3((unsigned)(p.rpc * p.tpr));
    cfg.dynamicSmemBytes = (size_t)dynamic_smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)p.cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, k, a);
}

// dt: DT_BF16 or DT_F16, the 16-bit activation type.
cudaError_t launch_norm(int fmt, int dt, const Plan& p, const NormArgs& a, cudaStream_t stream);
cudaError_t launch_norm_f16(int fmt, const Plan& p, const NormArgs& a, cudaStream_t stream);
// The persistent per-token norm (exact-fit plans, quantised output).
cudaError_t launch_norm_pt_persistent(int dt, const Plan& p, const NormArgs& a, cudaStream_t stream);
cudaError_t launch_norm_pt_persistent_f16(const Plan& p, const NormArgs& a, cudaStream_t stream);
// p.grid covers both segments; p.rpc * p.tpr is the common CTA size.
cudaError_t launch_norm_dual(int fmt, int dt, const Plan& p, const DualArgs& d, cudaStream_t stream);

// Records the CUDA error of a failed launch for sgq_launch_error() (per thread).
void note_launch_error(cudaError_t e);
// clamp16: the OAI kernels that clamp on packed bf16 (see swiglu_quant_kernel).
cudaError_t launch_swiglu(int fmt, const Plan& p, const SwigluArgs& a, bool clamp16, cudaStream_t stream);
cudaError_t launch_swiglu_oai_full(int fmt, const Plan& p, const SwigluArgs& a, bool clamp16, cudaStream_t stream);
cudaError_t launch_swiglu_oai_part(int fmt, const Plan& p, const SwigluArgs& a, bool clamp16, cudaStream_t stream);
cudaError_t launch_swiglu_silu_full(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream);
cudaError_t launch_swiglu_silu_part(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream);
cudaError_t launch_quant(int fmt, int dt, const Plan& p, const QuantArgs& a, cudaStream_t stream);

// The norm with the all-reduce of aa.ar.n partial inputs folded in (bf16).
cudaError_t launch_norm_ar(int fmt, const Plan& p, const NormARArgs& aa, cudaStream_t stream);

// Rows wider than one CTA covers, split over a cluster of p.cluster CTAs a
// row (p.grid = rows * p.cluster, p.rpc = 1, four chunks a thread).
cudaError_t launch_norm_cluster(int fmt, int dt, const Plan& p, const NormArgs& a, cudaStream_t stream);
cudaError_t launch_swiglu_pt_cluster(const Plan& p, const SwigluArgs& a, bool clamp16, cudaStream_t stream);
cudaError_t launch_quant_pt_cluster(int dt, const Plan& p, const QuantArgs& a, cudaStream_t stream);

}  // namespace sgq
