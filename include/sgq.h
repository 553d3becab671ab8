/*
 * sgq.h -- fused pre-GEMM activation epilogue for NVIDIA GB300 (sm_103a).
 *
 * Two fused operations, each one CUDA kernel launch on the caller's stream:
 *
 *   rmsnorm_add_quant  residual add + RMSNorm + FP8 activation quantisation
 *                      (+ optional bf16 copy of the normed rows)
 *   swiglu_quant       fp32 SwiGLU (OAI clamped, or SiLU-and-mul)
 *                      + the same quantisation
 *
 * and the three steps of the unfused chains they replace, also one launch
 * each, so that "norm, then a separate quant" and "activation, then a
 * separate quant" can be run and timed beside the fused forms:
 *
 *   rmsnorm_add        residual add + RMSNorm to bf16
 *   swiglu             SwiGLU to bf16
 *   quantize_fp8       FP8 quantisation of bf16 rows
 *
 * and a two-segment norm, one launch for two row sets over the same rows:
 *
 *   rmsnorm_dual_quant the q and kv latent norms of multi-head latent
 *                      attention (each segment quantised and/or copied)
 *
 * and the tensor-parallel all-reduce folded into the fused norm:
 *
 *   allreduce_rmsnorm_add_quant  the ranks' partial rows summed, then
 *                      residual add + RMSNorm + FP8 quantisation
 *
 * The operations follow these pages:
 *   [P1] "[ROCm][MiniMax-M3.1] Fuse MXFP8 quant into the add+RMSNorm and
 *        SwiGLU epilogues" (vllm PR 65478): "Purpose" (the two fusions),
 *        "Test Plan / Correctness" (bit-identical norm, fp32-direct SwiGLU),
 *        review "Scale layout / scheme contract" (row-major, unswizzled
 *        [M, N/32] E8M0 scales).
 *   [P2] "[Perf] [AMD] qwen3: Fuse the 1x128 FP8 input quant into RMSNorm
 *        and SiLU-and-mul" (sglang PR 48043): "Modifications" (1x128 group
 *        FP8; SiLU-and-mul rounded like the unfused op; bf16 inputs only).
 *   [P4] "[ROCm] Fuse per-token activation quant into RMSNorm" (sglang PR
 *        34502): "Change" (per-token FP8, [m, 1] scale; fp16 activations
 *        stay fp16; the q/kv norm), "Motivation" (the standalone quant).
 *
 * Conventions shared by all entry points
 *   - All tensor pointers are DEVICE pointers owned by the caller (the dual
 *     norm's two segment descriptors are host structs, read during the call
 *     only). The library allocates nothing, never synchronises and launches
 *     nothing but its one kernel, so calls may be captured into CUDA graphs.
 *     State kept between calls: the calling thread's last launch error (see
 *     sgq_launch_error), each device's multiprocessor count (queried on the
 *     first call on that device), the shared-memory opt-in each kernel was
 *     given on each device, the occupancy calculator's answer for each
 *     persistent launch shape (asked on its first launch), and the planning
 *     count of sgq_set_sm_budget.
 *   - All tensors are contiguous and row-major (the dual norm's inputs may
 *     have a row stride). 16-bit activations are bfloat16, or IEEE fp16 with
 *     SGQ_F_FP16 where an entry point accepts it. Quantised values are OCP
 *     E4M3 ("e4m3fn") bytes.
 *   - Scale layouts: MXFP8 -> uint8 E8M0 codes [M, W/32] (value 2^(code-127));
 *     1x128 block -> float32 [M, W/128]; per-token -> float32 [M, 1]; all
 *     row-major unless a layout flag below selects another one.
 *   - Alignment: every tensor pointer must be 16-byte aligned, except a
 *     float32 scale pointer (4 bytes) and an E8M0 scale pointer (1 byte).
 *   - Width rules: MXFP8 needs W % 32 == 0, 1x128 needs W % 128 == 0,
 *     per-token (and the unquantised outputs of rmsnorm_add, swiglu and an
 *     unquantised dual segment) needs W % 8 == 0; W <= SGQ_MAX_WIDTH
 *     (SGQ_MAX_DUAL_WIDTH for rmsnorm_dual_quant and
 *     allreduce_rmsnorm_add_quant).
 *   - Outputs may not overlap inputs or each other, except that residual_out
 *     may equal residual_in exactly (in-place update).
 *   - Launch order: every kernel may begin while the kernel before it on the
 *     stream is finishing (programmatic dependent launch), and waits for
 *     that kernel to complete before it reads an activation or writes any
 *     output. The norms read their weight before that wait, so the kernel
 *     launched just before a norm on its stream must not write that norm's
 *     weight (weights written by a copy, or by any earlier kernel, are fine).
 *   - M == 0 returns SGQ_OK without a launch (pointers are not inspected).
 *   - Errors: arguments are checked on the host before anything is launched;
 *     a rejected call leaves every buffer untouched. SGQ_ERR_LAUNCH reports a
 *     failed launch (the error cudaLaunchKernelEx returns for this launch; an
 *     error pending on the thread from other work is left alone).
 *   - Non-finite inputs (inf, NaN) are outside the contract: the kernels do
 *     not fault on them, but their outputs are unspecified. So are norm rows
 *     whose sum of squares overflows fp32 (|h| of order 1e19 / sqrt(H)).
 */
#ifndef SGQ_H
#define SGQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SGQ_ABI_VERSION 3
/* Widest row: rows up to 16384 columns run one CTA a row (or several, each a
 * column segment, at small M); wider rows run as a cluster of up to 8 CTAs,
 * or as column segments where no row-wide value is needed. */
#define SGQ_MAX_WIDTH 131072
/* Widest segment of rmsnorm_dual_quant, and widest row of
 * allreduce_rmsnorm_add_quant (rows no wider than one CTA covers). */
#define SGQ_MAX_DUAL_WIDTH 16384
/* Most partial inputs (tensor-parallel ranks) of allreduce_rmsnorm_add_quant. */
#define SGQ_MAX_RANKS 8

/* Quantisation format of the output activation. */
typedef enum sgq_format {
    SGQ_FMT_MXFP8 = 0,          /* E4M3 + one E8M0 scale per 1x32 block [P1] */
    SGQ_FMT_FP8_BLOCK128 = 1,   /* E4M3 + one fp32 scale amax/448 per 1x128 block [P2] */
    SGQ_FMT_FP8_PER_TOKEN = 2   /* E4M3 + one fp32 scale amax/448 per row [P4] */
} sgq_format_t;

/* Activation of swiglu_quant. */
typedef enum sgq_act {
    SGQ_ACT_SWIGLU_OAI = 0,     /* min(g,L) * sigmoid(alpha*min(g,L)) * (clamp(u,-L,L) + beta) [P1] */
    SGQ_ACT_SILU_MUL = 1        /* g * sigmoid(g) * u [P2] */
} sgq_act_t;

/* Flags. */
#define SGQ_F_GEMMA_WEIGHT    (1u << 0) /* norm: scale by (1 + w) (Gemma) instead of w */
#define SGQ_F_QUANT_FROM_FP32 (1u << 1) /* quantise the fp32 value, not its bf16 rounding */
#define SGQ_F_ACT_ROUND_BF16  (1u << 2) /* SiLU-and-mul: round silu(g) to bf16 before the product */
#define SGQ_F_FP16            (1u << 5) /* norms and quantize_fp8: the 16-bit activations (inputs,
                                           weight, written residual and normed rows, and the
                                           rounded quant source) are IEEE fp16, not bf16 */

/*
 * Scale layouts for GEMM consumers other than the row-major one. [P1]'s
 * review ("Scale layout / scheme contract") separates consumers that read
 * row-major [M, N/32] E8M0 scales from those that want them swizzled; these
 * flags give the layouts that Blackwell-class consumers read. Accepted by
 * rmsnorm_add_quant, swiglu_quant and quantize_fp8.
 *
 * SGQ_F_SCALE_SWIZZLED (MXFP8 only): the E8M0 codes in the tiled layout of
 *   block-scaled MMA operands (the scale-factor layout that cuBLASLt's
 *   VEC32_UE8M0 block scaling reads). Rows are padded to Mp = M rounded up
 *   to 128 and scale columns to Gp = W/32 rounded up to 4. The [Mp, Gp] codes
 *   are cut into 128 x 4 tiles of 512 bytes, stored tile-row by tile-row
 *   ((r/128) * (Gp/4) + g/4); inside a tile, row r and column g sit at byte
 *   (r % 32) * 16 + ((r / 32) % 4) * 4 + g % 4. Buffer: Mp * Gp bytes. The
 *   padding (rows >= M, columns >= W/32) is written as code 0.
 * SGQ_F_SCALE_COL_MAJOR (1x128 only): the fp32 scales column-major (group-
 *   major): scale (r, g) at g * Mp + r with Mp = M rounded up to 4, so every
 *   column starts 16-byte aligned from the base. Buffer: (W/128) * Mp * 4
 *   bytes. Rows >= M are written as 0.0f.
 * Either flag with another format is SGQ_ERR_INVALID_ARG.
 */
#define SGQ_F_SCALE_SWIZZLED  (1u << 3)
#define SGQ_F_SCALE_COL_MAJOR (1u << 4)

typedef enum sgq_status {
    SGQ_OK = 0,
    SGQ_ERR_INVALID_ARG = 1,    /* NULL required pointer, bad enum/flag, negative size, overlap */
    SGQ_ERR_UNSUPPORTED = 2,    /* width not a multiple of the group, or above the widest row */
    SGQ_ERR_MISALIGNED = 3,     /* a pointer breaks the alignment rule above */
    SGQ_ERR_LAUNCH = 4          /* the CUDA launch failed */
} sgq_status_t;

/* A cudaStream_t (NULL selects the legacy default stream). */
typedef void* sgq_stream_t;

/*
 * Residual add + RMSNorm + FP8 quantisation, one pass per row ([P1] "Purpose",
 * commit 1; [P2] "Modifications"; [P4] "Change"). For each row i:
 *
 *   h   = x[i] + residual_in[i]            (fp32; h = x[i] if residual_in is NULL)
 *   residual_out[i] = bf16(h)              (if residual_out is not NULL)
 *   inv = 1 / sqrt(sum_j h_j^2 / H + eps)
 *   y   = h * inv * (1 + w)  with SGQ_F_GEMMA_WEIGHT, else h * inv * w
 *   normed_out[i] = bf16(y)                (if normed_out is not NULL)
 *   src = y with SGQ_F_QUANT_FROM_FP32, else bf16(y)
 *   q_out[i], scale_out[i] = quantise(src) in format fmt
 *
 * Quantisation of one group (32, 128 or H elements) with amax = max |src|:
 *   MXFP8: e = clamp(floor(log2(amax)) - 8, -127, 127) (amax = 0 -> -127);
 *          scale code = e + 127; q = E4M3_rn_satfinite(src * 2^-e).
 *   FP8:   s = fp32(amax / 448); q = E4M3_rn_satfinite(fp32(src / s));
 *          s = 0 gives q = 0.
 *
 * Arguments:
 *   fmt           sgq_format_t
 *   flags         SGQ_F_GEMMA_WEIGHT | SGQ_F_QUANT_FROM_FP32 | SGQ_F_FP16, and a
 *                 scale layout flag of the format (others rejected). With
 *                 SGQ_F_FP16 the bf16 of the formulas above reads fp16.
 *   M, H          rows and hidden width
 *   eps           >= 0, finite; with eps = 0 a row whose h is all zero has no
 *                 defined result (1/sqrt(0); its outputs are unspecified)
 *   x             [M, H] bf16, read
 *   residual_in   [M, H] bf16, read, or NULL
 *   residual_out  [M, H] bf16, written, or NULL; must be NULL when residual_in
 *                 is NULL; may equal residual_in
 *   weight        [H] bf16, read before the launch waits for the kernel that
 *                 precedes it on the stream, which must not write it (see
 *                 "Launch order" above)
 *   q_out         [M, H] E4M3, written
 *   scale_out     scales in the layout of fmt and flags, written
 *   normed_out    [M, H] bf16, written, or NULL
 *   stream        the stream to launch on
 */
int rmsnorm_add_quant(int fmt, uint32_t flags, int64_t M, int64_t H, float eps,
                      const void* x, const void* residual_in, void* residual_out,
                      const void* weight, void* q_out, void* scale_out, void* normed_out,
                      sgq_stream_t stream);

/*
 * Tensor-parallel all-reduce + residual add + RMSNorm + FP8 quantisation in
 * one launch ([P1] "Purpose" commit 1, the all-reduce + norm entry point, and
 * "Limitations", a quant-emitting fused all-reduce + norm; [P4] "Change", the
 * fused all-reduce + RMSNorm + quant of the entry projection). Each of the
 * nranks ranks of a tensor-parallel group holds a partial [M, H] bf16 result
 * of the preceding row-parallel GEMM; the all-reduce's output is their sum.
 * For each row i:
 *
 *   x   = bf16(partials[0][i] + partials[1][i] + ... )   (fp32, in rank order)
 *   then exactly rmsnorm_add_quant of x, residual_in, weight.
 *
 * So the result equals rmsnorm_add_quant applied to that x, bit for bit.
 * "One shot": every rank calls it over all M rows, reading every rank's
 * partial. "Two shot": each rank calls it on its own slice of rows (pointers
 * offset by the slice's first row, M = the slice's rows), then the ranks
 * gather the slices' outputs (the quantised rows are half the bf16 bytes).
 *
 * Arguments as for rmsnorm_add_quant, except:
 *   flags         SGQ_F_GEMMA_WEIGHT | SGQ_F_QUANT_FROM_FP32 and a scale layout
 *                 flag of the format (bf16 activations only)
 *   nranks        1 .. SGQ_MAX_RANKS
 *   H             a multiple of the format's group, at most SGQ_MAX_DUAL_WIDTH
 *   partials      HOST array of nranks DEVICE pointers, each [M, H] bf16, read;
 *                 on a multi-GPU node these may be other GPUs' memory mapped
 *                 into this one (peer access), read with plain loads. The
 *                 caller makes every partial complete and visible before the
 *                 launch begins (e.g. a barrier among the ranks): the kernel
 *                 waits for nothing. Partials may overlap each other and the
 *                 inputs; no output may overlap any of them.
 * SGQ_ERR_UNSUPPORTED also when the staging of nranks partials would need
 * more shared memory than a CTA has (wide rows with many ranks).
 */
int allreduce_rmsnorm_add_quant(int fmt, uint32_t flags, int nranks, int64_t M, int64_t H, float eps,
                                const void* const* partials, const void* residual_in, void* residual_out,
                                const void* weight, void* q_out, void* scale_out, void* normed_out,
                                sgq_stream_t stream);

/*
 * SwiGLU + FP8 quantisation, one pass per row ([P1] "Purpose", commit 2 and
 * "Test Plan / Correctness"; [P2] "Modifications"). gate_up is [M, 2I] bf16:
 * gate g = columns [0, I), up u = columns [I, 2I). For each element:
 *
 *   OAI:  g' = min(g, limit); u' = min(max(u, -limit), limit);
 *         a = g' * sigmoid(alpha * g') * (u' + beta)       (fp32)
 *   SiLU: a = silu(g) * u, silu(g) = g * sigmoid(g)       (fp32); with
 *         SGQ_F_ACT_ROUND_BF16 silu(g) is rounded to bf16 before the product
 *   src = a with SGQ_F_QUANT_FROM_FP32, else bf16(a)
 *   q_out, scale_out = quantise(src) as for rmsnorm_add_quant.
 *
 * [P1]'s fused OAI SwiGLU quantises the fp32 value (SGQ_F_QUANT_FROM_FP32);
 * [P2]'s SiLU-and-mul rounds like the unfused op (SGQ_F_ACT_ROUND_BF16 and
 * no SGQ_F_QUANT_FROM_FP32).
 *
 * Arguments:
 *   fmt, act      sgq_format_t, sgq_act_t
 *   flags         SGQ_F_QUANT_FROM_FP32, SGQ_F_ACT_ROUND_BF16 with
 *                 SGQ_ACT_SILU_MUL only, and a scale layout flag of the
 *                 format (others rejected)
 *   M, I          rows and intermediate width (the output width)
 *   alpha, beta, limit  OAI parameters (finite alpha and beta, limit > 0,
 *                 may be +inf); ignored for SiLU-and-mul
 *   gate_up       [M, 2I] bf16, read
 *   q_out         [M, I] E4M3, written
 *   scale_out     scales in the layout of fmt and flags, written
 *   stream        the stream to launch on
 */
int swiglu_quant(int fmt, int act, uint32_t flags, int64_t M, int64_t I, float alpha,
                 float beta, float limit, const void* gate_up, void* q_out, void* scale_out,
                 sgq_stream_t stream);

/*
 * Residual add + RMSNorm to bf16 alone: the first step of the unfused chain
 * "norm, then a separate quant" that [P1] "Microbenchmark script" times
 * against the fused kernel, and that [P2] "Modifications" and [P4]
 * "Motivation" describe (the quant ran as its own launch after the norm).
 * Computes h, residual_out and normed_out exactly as rmsnorm_add_quant does;
 * writes no quantised output. quantize_fp8(normed_out) then equals
 * rmsnorm_add_quant without SGQ_F_QUANT_FROM_FP32, byte for byte.
 *
 * Arguments as for rmsnorm_add_quant, except:
 *   flags         SGQ_F_GEMMA_WEIGHT | SGQ_F_FP16 (others rejected)
 *   H             any multiple of 8 up to SGQ_MAX_WIDTH
 *   normed_out    [M, H] bf16, written (required)
 */
int rmsnorm_add(uint32_t flags, int64_t M, int64_t H, float eps, const void* x,
                const void* residual_in, void* residual_out, const void* weight,
                void* normed_out, sgq_stream_t stream);

/*
 * SwiGLU to bf16 alone: the first step of the unfused chain "activation,
 * then a separate quant" ([P1] "Microbenchmark script"; [P2]
 * "Modifications"). out = bf16(a), a the fp32 activation of swiglu_quant
 * (with SGQ_F_ACT_ROUND_BF16, silu(g) rounded to bf16 before the product).
 * quantize_fp8(out) then equals swiglu_quant without SGQ_F_QUANT_FROM_FP32,
 * byte for byte.
 *
 * Arguments as for swiglu_quant, except:
 *   flags         SGQ_F_ACT_ROUND_BF16 with SGQ_ACT_SILU_MUL only
 *   I             any multiple of 8 up to SGQ_MAX_WIDTH
 *   out           [M, I] bf16, written
 */
int swiglu(int act, uint32_t flags, int64_t M, int64_t I, float alpha, float beta,
           float limit, const void* gate_up, void* out, sgq_stream_t stream);

/*
 * FP8 quantisation of bf16 rows alone, in any of the three formats: the
 * separate quant launch of the unfused chains ([P1] "Purpose" and
 * "Microbenchmark script"; [P2] "Modifications"; [P4] "Motivation").
 * q_out, scale_out = quantise(src) with the group rule of rmsnorm_add_quant.
 *
 * Arguments:
 *   fmt           sgq_format_t
 *   flags         SGQ_F_FP16 (src is fp16), and a scale layout flag of the
 *                 format (others rejected)
 *   M, W          rows and width (W a multiple of the group, <= SGQ_MAX_WIDTH)
 *   src           [M, W] bf16, read
 *   q_out         [M, W] E4M3, written
 *   scale_out     scales in the layout of fmt and flags, written
 *   stream        the stream to launch on
 */
int quantize_fp8(int fmt, uint32_t flags, int64_t M, int64_t W, const void* src, void* q_out,
                 void* scale_out, sgq_stream_t stream);

/* One row set of rmsnorm_dual_quant. */
typedef struct sgq_norm_seg {
    int64_t H;             /* width */
    int64_t ld;            /* row stride of x in elements: >= H, a multiple of 8 */
    const void* x;         /* rows of x: [M, ld] 16-bit, columns [0, H) read */
    const void* weight;    /* [H] 16-bit */
    void* q_out;           /* [M, H] E4M3, or NULL: this segment is not quantised */
    void* scale_out;       /* scales of fmt (row-major), NULL exactly when q_out is */
    void* normed_out;      /* [M, H] 16-bit normed rows, or NULL (not with q_out NULL) */
} sgq_norm_seg_t;

/*
 * Two RMSNorms over the same M rows in one launch, each with its own input
 * rows, weight and outputs, and no residual: the q and kv latent norms of
 * multi-head latent attention ([P4] "Change": the decode q_b_proj quant is
 * folded into the fused q/kv RMSNorm, which emits the per-token quantised q
 * while kv stays in the activation type). For each segment, each row:
 *
 *   y = x * inv * (1 + w) (SGQ_F_GEMMA_WEIGHT) or x * inv * w,
 *   inv = 1 / sqrt(sum_j x_j^2 / H + eps)
 *   normed_out = 16-bit(y)                  (if normed_out is not NULL)
 *   q_out, scale_out = quantise(src)        (if q_out is not NULL)
 *
 * exactly as rmsnorm_add_quant computes a row without residual, so each
 * segment's outputs equal a rmsnorm_add_quant call on its rows, bit for bit
 * (each segment keeps that call's threads per row). The one exception: width
 * pairs whose single-norm threads per row have a least common multiple above
 * 512 (for instance 7168 and 2240 at small M) run both segments at one
 * width's threads per row, and then match a single call within the parity
 * tolerances. The inputs
 * may be column ranges of one tensor (x = base + column offset, ld = the
 * tensor's row length), and may overlap each other; the outputs may overlap
 * nothing. Scales are row-major (no layout flags).
 *
 * Arguments:
 *   fmt           sgq_format_t (both segments)
 *   flags         SGQ_F_GEMMA_WEIGHT | SGQ_F_QUANT_FROM_FP32 | SGQ_F_FP16
 *   M             rows of both segments
 *   eps           >= 0, finite (eps = 0 and an all-zero row: as rmsnorm_add_quant)
 *   seg_a, seg_b  host pointers to the two segments (read during the call
 *                 only); H a multiple of the format's group when the segment
 *                 is quantised, else of 8; H <= SGQ_MAX_DUAL_WIDTH
 *   stream        the stream to launch on
 */
int rmsnorm_dual_quant(int fmt, uint32_t flags, int64_t M, float eps, const sgq_norm_seg_t* seg_a,
                       const sgq_norm_seg_t* seg_b, sgq_stream_t stream);

/*
 * Plan launches as if the device had `sms` multiprocessors; 0 (the default)
 * uses the current device's own count, queried once per device. The count
 * decides how many rows share a CTA, how many threads own a row and when a
 * row runs as several CTAs (column segments), e.g. for callers that give
 * these kernels only part of the GPU (an MPS or green-context partition).
 * Every plan meets the same contract, but a norm's sum of squares is added
 * in the order its plan gives, so the bits of a norm's outputs may differ
 * between two counts (within the stated tolerances of the definition).
 * Process-wide, for calls made after it returns. sms < 0 returns
 * SGQ_ERR_INVALID_ARG. Not part of any page: a host planning control.
 */
int sgq_set_sm_budget(int sms);

/* A static, human-readable name of a status code. */
const char* sgq_status_string(int status);

/* SGQ_ABI_VERSION of the loaded library. */
int sgq_abi_version(void);

/* The CUDA error text of the calling thread's most recent call that returned
 * SGQ_ERR_LAUNCH ("no launch error" if there was none). Static storage. */
const char* sgq_launch_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SGQ_H */
