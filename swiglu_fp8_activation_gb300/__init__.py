"""Fused pre-GEMM activation epilogue for NVIDIA GB300 (sm_103a).

Two fused ops behind a C ABI (`libsgq.so`, declared in include/sgq.h):

* `rmsnorm_add_quant`: residual add + RMSNorm (Gemma `(1+w)` or plain `w`)
  + FP8 activation quantisation, with an optional bf16 copy of the normed rows.
* `swiglu_quant`: fp32 SwiGLU (OAI clamped, or SiLU-and-mul) + the same
  quantisation.

The three steps of the unfused chains they replace are exported too, one
launch each, to run and time beside them: `rmsnorm_add` (norm to bf16),
`swiglu` (activation to bf16) and `quantize_fp8` (FP8 quant of bf16 rows).
`rmsnorm_dual_quant` norms two row sets (the q and kv latent norms) in one
launch, and `allreduce_rmsnorm_add_quant` folds a tensor-parallel all-reduce
(the ranks' partial rows summed in rank order) into the fused norm; the `tp`
module holds its two-shot row partition and gather. The norms and the quant
also take fp16 activations.

Formats: MXFP8 (E4M3 + one E8M0 scale per 1x32 block), 1x128 block FP8 with
fp32 scales, and per-token FP8 with an [M,1] fp32 scale.

The CUDA library is loaded on first use; a missing library raises an error
(there is no CPU fallback).
"""
from .binding import (  # noqa: F401
    FORMATS, ACTS, F_GEMMA_WEIGHT, F_QUANT_FROM_FP32, F_ACT_ROUND_BF16, F_SCALE_SWIZZLED, F_SCALE_COL_MAJOR,
    SCALE_LAYOUTS, scale_shape,
    SgqError, library, library_path, rmsnorm_add_quant, swiglu_quant, status_string,
    rmsnorm_add, swiglu, quantize_fp8, rmsnorm_dual_quant, NormSeg, F_FP16, set_sm_budget,
    allreduce_rmsnorm_add_quant, MAX_RANKS,
)
