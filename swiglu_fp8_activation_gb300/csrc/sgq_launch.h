// sgq_launch.h -- host-side launchers of the row-engine kernels (one
// translation unit per operation, so they compile in parallel).
#pragma once

#include <cuda_runtime.h>

#include "sgq_kernels.cuh"

namespace sgq {

// Launch geometry of one call: `nv` chunks per thread, `tpr` threads per row,
// `rpc` rows per CTA, `grid` CTAs.
struct Plan {
    int nv;
    int tpr;
    int rpc;
    int64_t grid;
};

// Pick a plan for M rows of width W (W % 8 == 0). Returns false when W needs
// more than kMaxTPR threads per row.
bool plan_rows(int64_t M, int W, int sm_count, Plan* p);

cudaError_t launch_norm(int fmt, const Plan& p, const NormArgs& a, cudaStream_t stream);
cudaError_t launch_swiglu(int fmt, const Plan& p, const SwigluArgs& a, cudaStream_t stream);

}  // namespace sgq
