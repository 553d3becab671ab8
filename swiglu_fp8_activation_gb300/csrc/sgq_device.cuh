// sgq_device.cuh -- device code of the fused norm / SwiGLU + FP8 quantisation
// kernels for sm_103a.
//
// One "row engine" serves every operation. A row of W elements is split into
// 16-byte chunks of 8 16-bit values; `tpr` threads (a multiple of 32) own one
// row, and thread t owns chunks t, t + tpr, ..., t + (NV-1)*tpr, so every
// warp-wide copy is 512 contiguous bytes. All NV chunks of a thread are copied
// asynchronously into its own shared-memory slots before any arithmetic (one
// commit group per chunk), so the whole row is in flight without holding
// registers, and each chunk is processed as soon as its group has landed; the
// row is read from global memory once. Reductions:
//   * sum of squares (RMSNorm) and per-token amax: warp shuffles, then one
//     shared-memory step across the row's warps;
//   * 1x32 (MX) amax: the 4 lanes that own one 32-block (2 xor-shuffles);
//   * 1x128 amax: the 16 lanes that own one 128-block (4 xor-shuffles).
// Block alignment holds because tpr is a multiple of 32 and W is a multiple
// of the group size: chunk c lives in lane c % 32 of its warp, so a 32-block
// (4 chunks) or a 128-block (16 chunks) never straddles a lane group.
//
// Numeric formats: bf16 = upper half of IEEE binary32; fp16 = IEEE binary16;
// E4M3 = OCP "e4m3fn"; E8M0 = OCP MX scale byte, value 2^(code-127). The
// operations follow
// "[ROCm][MiniMax-M3.1] Fuse MXFP8 quant into the add+RMSNorm and SwiGLU
// epilogues" (vllm PR 65478, "Purpose"), "[Perf] [AMD] qwen3: Fuse the 1x128
// FP8 input quant into RMSNorm and SiLU-and-mul" (sglang PR 48043,
// "Modifications") and "[ROCm] Fuse per-token activation quant into RMSNorm"
// (sglang PR 34502, "Change").
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sgq {

enum Fmt : int { FMT_MX = 0, FMT_B128 = 1, FMT_PT = 2 };
enum Act : int { ACT_OAI = 0, ACT_SILU = 1 };
enum ScaleLayout : int { SCALE_ROW_MAJOR = 0, SCALE_SWIZZLED = 1, SCALE_COL_MAJOR = 2 };
enum IoType : int { DT_BF16 = 0, DT_F16 = 1 };   // the 16-bit activation type

constexpr uint32_t F_GEMMA = 1u << 0;
constexpr uint32_t F_FROM_FP32 = 1u << 1;
constexpr uint32_t F_ACT_BF16 = 1u << 2;

constexpr int kMaxNV = 4;          // chunks per thread
constexpr int kMaxTPR = 512;       // threads per row (one CTA covers kMaxTPR * kMaxNV * 8 columns)
constexpr int kTargetCTA = 256;    // threads per CTA when several rows share one
constexpr int kMaxCluster = 8;     // CTAs a row at most when a row is wider than one CTA covers
constexpr int kMaxRanks = 8;       // partial inputs of the all-reduce folded into the norm

// ----------------------------------------------------------------- memory

// 16-byte asynchronous copy from global to shared memory, caching in L2 only
// (with a 256-byte L2 prefetch). src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes)
                 : "memory");
}

// The same, allocating in L1 as well: for data every row of the SM reads (the norm weight).
__device__ __forceinline__ void cp_async16_cached(void* smem, const void* gmem, int src_bytes) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's committed copy groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// With NV groups committed in order, wait for group v (v is a constant after unrolling).
template <int NV>
__device__ __forceinline__ void cp_async_wait_group_of(int v) {
    const int pending = NV - 1 - v;
    if (pending >= 7) cp_async_wait<7>();
    else if (pending == 6) cp_async_wait<6>();
    else if (pending == 5) cp_async_wait<5>();
    else if (pending == 4) cp_async_wait<4>();
    else if (pending == 3) cp_async_wait<3>();
    else if (pending == 2) cp_async_wait<2>();
    else if (pending == 1) cp_async_wait<1>();
    else cp_async_wait<0>();
}

__device__ __forceinline__ uint4 ld_smem16(const uint4* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
    return v;
}

// Global stores of kernel outputs, predicated in PTX (no branch around them).
// Nothing in these kernels reads an output back, so no memory clobber.
__device__ __forceinline__ void st16_if(void* p, uint4 v, bool pred) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %5, 0;\n\t@p st.global.v4.u32 [%0], {%1,%2,%3,%4};\n}" ::"l"(p),
        "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"((int)pred));
}

// The same with the streaming (evict-first) cache policy, for an output that
// no kernel soon after reads back, so that its lines leave L2 for memory
// first and do not linger dirty into the next kernel's time.
__device__ __forceinline__ void st16_cs_if(void* p, uint4 v, bool pred) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %5, 0;\n\t@p st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};\n}" ::"l"(p),
        "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"((int)pred));
}

__device__ __forceinline__ void st8_if(void* p, uint2 v, bool pred) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %3, 0;\n\t@p st.global.v2.u32 [%0], {%1,%2};\n}" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"((int)pred));
}

__device__ __forceinline__ void st_u8_if(void* p, uint32_t v, bool pred) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t@p st.global.u8 [%0], %1;\n}" ::"l"(p), "r"(v),
                 "r"((int)pred));
}

__device__ __forceinline__ void st_f32_if(void* p, float v, bool pred) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t@p st.global.f32 [%0], %1;\n}" ::"l"(p), "f"(v),
                 "r"((int)pred));
}

// ------------------------------------------------------------ conversions

// 8 bf16 (one chunk) -> 8 floats; element k sits in bits [16k, 16k+16) of the chunk.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Elementwise min / max of two bf16x2 pairs (finite values: exact).
__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two floats -> bf16x2 with round-to-nearest-even; `lo` goes to the low half.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint4 f32x8_to_bf16x8(const float f[8]) {
    return make_uint4(f32x2_to_bf16x2(f[0], f[1]), f32x2_to_bf16x2(f[2], f[3]),
                      f32x2_to_bf16x2(f[4], f[5]), f32x2_to_bf16x2(f[6], f[7]));
}

// Round two floats to the nearest bf16 (ties to even) and widen them back:
// one conversion for the pair.
__device__ __forceinline__ float2 round_bf16x2(float2 v) {
    const uint32_t p = f32x2_to_bf16x2(v.x, v.y);
    return make_float2(__uint_as_float(p << 16), __uint_as_float(p & 0xFFFF0000u));
}

// Round a float to the nearest bf16 (ties to even) and widen it back.
__device__ __forceinline__ float round_bf16(float v) {
    return __uint_as_float(f32x2_to_bf16x2(v, 0.0f) << 16);
}

// fp16x2 (low half first) -> two floats (exact).
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t w) {
    float lo, hi;
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
    return make_float2(lo, hi);
}

// Two floats -> fp16x2 with round-to-nearest-even; `lo` goes to the low half.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Eight 16-bit values of type DT (one 16-byte chunk) -> floats, and back
// with round-to-nearest-even; round_io rounds one float to DT and widens it.
template <int DT>
__device__ __forceinline__ void load8(const uint4 v, float f[8]) {
    if (DT == DT_BF16) {
        bf16x8_to_f32(v, f);
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = f16x2_to_f32x2(w[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
}

template <int DT>
__device__ __forceinline__ uint4 pack8(const float f[8]) {
    if (DT == DT_BF16) return f32x8_to_bf16x8(f);
    return make_uint4(f32x2_to_f16x2(f[0], f[1]), f32x2_to_f16x2(f[2], f[3]), f32x2_to_f16x2(f[4], f[5]),
                      f32x2_to_f16x2(f[6], f[7]));
}

template <int DT>
__device__ __forceinline__ float round_io(float v) {
    if (DT == DT_BF16) return round_bf16(v);
    return f16x2_to_f32x2(f32x2_to_f16x2(v, 0.0f)).x;
}

// Four floats -> four E4M3 bytes (round to nearest even, saturate to +-448);
// element 0 goes to the lowest byte.
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float a0, float a1, float a2, float a3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a1), "f"(a0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(a3), "f"(a2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// ------------------------------------------------------- launch ordering

// Programmatic dependent launch. pdl_wait() blocks until the grid this launch
// depends on has completed and its writes are visible; it returns at once
// when the launch has no programmatic dependency. Every kernel here calls it
// before it reads an activation or writes anything; only the norms' weight,
// which the entry points require the preceding kernel not to write, is read
// before it.
// pdl_trigger() lets the next grid on the stream begin launching; that grid
// in turn waits in its own pdl_wait() before touching memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- clusters

// Thread block clusters: the CTAs of a cluster run at the same time, and each
// may write the others' shared memory. A row wider than one CTA covers is
// split over the CTAs of one cluster, which exchange their partial reductions
// through shared memory (no global memory, no flags).
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_ctas() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// The cluster barrier in two halves: every thread of every CTA of the
// cluster arrives, then waits for all the others (hardware barrier phases,
// as __syncthreads is for one CTA). The relaxed arrive orders no memory; the
// release / acquire pair makes the shared-memory stores before the arrive
// visible to the threads after the wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Store v into the copy of the shared variable at p held by the cluster's
// CTA `rank`.
__device__ __forceinline__ void st_cluster_f32x2(const void* p, uint32_t rank, float2 v) {
    const uint32_t local = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(v.x), "f"(v.y) : "memory");
}

// One float2 from every CTA of the cluster, combined in rank order (sum of
// .x, max of .y, which is >= 0), so that every CTA gets the bit-identical
// result. v is this CTA's value (the same in all its threads). Every thread
// of every CTA calls it once, after cluster_arrive_relaxed(): the wait that
// completes that arrive guarantees every CTA of the cluster is running
// before any thread writes another's shared memory; CTA i's thread j writes
// v into slot i of CTA j, and the second arrive / wait makes those stores
// visible. No shared memory of another CTA is touched afterwards, so each
// CTA may exit when it likes.
__device__ __forceinline__ float2 cluster_combine(float2 v, float2 (&slots)[kMaxCluster]) {
    const uint32_t n = cluster_ctas(), me = cluster_rank();
    cluster_wait();
    if (threadIdx.x < n) st_cluster_f32x2(&slots[me], threadIdx.x, v);
    cluster_arrive();
    cluster_wait();
    float2 r = slots[0];
    for (uint32_t i = 1; i < n; ++i) r = make_float2(r.x + slots[i].x, fmaxf(r.y, slots[i].y));
    return r;
}

// ------------------------------------------------------------ arithmetic

// Hardware reciprocal approximation (about 1 ulp); subnormal inputs and
// results flush to zero, which the callers never produce (they pass values
// in [1, 2]).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(e) split into an fp32 head (round to nearest) and the fp32 rounding of
// the remainder.
constexpr float kLog2eHi = 1.44269502162933349609375f;   // 0x3FB8AA3B
constexpr float kLog2eLo = 1.925963033500011e-08f;       // log2(e) - kLog2eHi
constexpr float kLn2 = 0.693147180559945309f;        // ln 2, rounded to fp32
constexpr float kInv448 = 0x1.24924ap-9f;             // 1/448 rounded to nearest fp32 (the FP8 scale divisor)

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Arguments z of the sigmoid must lie in [kSigLo, kSigHi] (callers clamp).
// Past kSigHi the sigmoid is 1.0 in fp32 (1 - e^-20 rounds to 1); below
// kSigLo it is 0 (e^-104 is below half the smallest fp32 subnormal).
constexpr float kSigLo = -104.0f, kSigHi = 20.0f;

// Logistic sigmoid 1/(1 + E), E = e^-z, of the 8 values of one chunk, for
// z = kz * x given as x and the negated scaled log2(e) split in fp32 parts:
// khi + klo = -kz log2(e) (kz = 1 for the plain sigmoid, alpha for OAI), so
// that E = 2^q with q = (khi + klo) x. Written from the mathematics on packed
// fp32x2 arithmetic:
//   * q is carried as the head qh = RN(khi x) plus a tail: the exact FMA
//     residual of that product and klo x, in the manner of Cody and Waite's
//     argument reduction; |tail| < 2^-16;
//   * the hardware 2^x takes the head, whose every value it evaluates to
//     about 2 ulp, and the tail enters to first order:
//     2^q = 2^qh (1 + tail ln 2), the dropped second-order term being below
//     2^-33 relative;
//   * sigmoid = 1/(1+E), the hardware reciprocal refined by one
//     Newton-Raphson step. Where qh > 125 (z < -86.6, a branch taken once
//     per chunk) 1/(1+E) would leave the normal range, and the sigmoid, then
//     2^-q to within 2^-125 relative, is formed as 2^(126-qh) (1 - tail ln 2)
//     scaled by 2^-126.
// Valid for any x with |q| below 2^120 whose z is at least kSigLo.
__device__ __forceinline__ void sigmoid8(const float (&x)[8], float khi, float klo, float (&out)[8]) {
    float2 e[4], m[4];
    float qmax = -1.0e30f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 xv = make_float2(x[2 * i], x[2 * i + 1]);
        const float2 qh = __fmul2_rn(xv, f2(khi));                       // head, rounded
        const float2 nr = __ffma2_rn(xv, f2(-khi), qh);                  // -(khi x - qh), exact
        const float2 nt = __ffma2_rn(xv, f2(-klo), nr);                  // -tail
        m[i] = __fmul2_rn(nt, f2(-kLn2));                                // 2^q = 2^qh (1 + m)
        e[i] = make_float2(ex2_approx(qh.x), ex2_approx(qh.y));
        qmax = fmaxf(qmax, fmaxf(qh.x, qh.y));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 E = __ffma2_rn(e[i], m[i], e[i]);
        const float2 d = __fadd2_rn(E, f2(1.0f));
        const float2 r0 = make_float2(rcp_approx(d.x), rcp_approx(d.y));
        // 1 - d*r0, with -d = RN(-(1 + E)) the exact negation of d (rounding to nearest is symmetric)
        const float2 res = __ffma2_rn(make_float2(-d.x, -d.y), r0, f2(1.0f));
        const float2 r = __ffma2_rn(r0, res, r0);                          // one Newton-Raphson step
        out[2 * i] = r.x;
        out[2 * i + 1] = r.y;
    }
    if (qmax > 125.0f) {         // sigmoid = 2^-q for those past qh = 125
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float qh = x[2 * i + j] * khi;
                if (qh > 125.0f) {
                    const float mj = j ? m[i].y : m[i].x;
                    const float v = ex2_approx(126.0f - qh);             // 2^(126 - qh), in [2^-24, 2]
                    out[2 * i + j] = fmaf(v, -mj, v) * 0x1p-126f;
                }
            }
        }
    }
}

// The same for gate values whose far-negative tail the caller detected on
// the packed bf16 inputs: `rare` is true when some x may have
// RN(khi x) > 125. Here x is not clamped from below, so where RN(khi x) > 125
// the main formula may overflow (to inf or NaN); only those elements are
// recomputed, as in sigmoid8, from max(x, xlo), xlo the x whose sigmoid
// argument is kSigLo (below it the sigmoid is 0 in fp32). Every result equals
// sigmoid8's for the argument max(x, xlo).
__device__ __forceinline__ void sigmoid8_prechecked(const float (&x)[8], float khi, float klo, float xlo, bool rare,
                                                    float (&out)[8]) {
    float2 e[4], m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 xv = make_float2(x[2 * i], x[2 * i + 1]);
        const float2 qh = __fmul2_rn(xv, f2(khi));
        const float2 nr = __ffma2_rn(xv, f2(-khi), qh);
        const float2 nt = __ffma2_rn(xv, f2(-klo), nr);
        m[i] = __fmul2_rn(nt, f2(-kLn2));
        e[i] = make_float2(ex2_approx(qh.x), ex2_approx(qh.y));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 E = __ffma2_rn(e[i], m[i], e[i]);
        const float2 d = __fadd2_rn(E, f2(1.0f));
        const float2 r0 = make_float2(rcp_approx(d.x), rcp_approx(d.y));
        const float2 res = __ffma2_rn(make_float2(-d.x, -d.y), r0, f2(1.0f));
        const float2 r = __ffma2_rn(r0, res, r0);
        out[2 * i] = r.x;
        out[2 * i + 1] = r.y;
    }
    if (rare) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float xc = fmaxf(x[j], xlo);
            const float qh = xc * khi;
            if (qh > 125.0f) {
                const float nt = fmaf(xc, -klo, fmaf(xc, -khi, qh));
                const float mj = nt * -kLn2;
                const float v = ex2_approx(126.0f - qh);
                out[j] = fmaf(v, -mj, v) * 0x1p-126f;
            }
        }
    }
}

// True when either bf16 half of a is below the same half of b.
__device__ __forceinline__ bool bf16x2_any_lt(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("{\n\t.reg .pred p, q;\n\tsetp.lt.bf16x2 p|q, %1, %2;\n\tor.pred p, p, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(a), "r"(b));
    return r != 0;
}

// a / b rounded to nearest even, given r = RN(1/b) (b and r normal). q0 = a*r
// is within one ulp of a/b; the remainder a - b*q0 is exact in one FMA, and
// q0 + rem*r rounded once is the correctly rounded quotient (Markstein's
// correction step: P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990). Results
// below the normal range may differ from IEEE division by an ulp. The
// remainder's FMA rounds down: being exact, its value is the same in any
// rounding direction, but for a = +-0 the sum +0 + -0 it forms is then -0,
// so that the correction keeps the sign of a zero quotient (-0 / b = -0, as
// in IEEE division; rounding to nearest would give +0).
__device__ __forceinline__ float div_rn(float a, float b, float r) {
    const float q0 = a * r;
    const float rem = __fmaf_rd(-q0, b, a);
    return fmaf(rem, r, q0);
}

// Two quotients at once, as div_rn, given nb = -b and r = RN(1/b) for the
// same b (one FP8 group's scale): q0 = a*r; rem = a - b*q0 (exact, rounded
// down for the sign of zero); q0 + rem*r.
__device__ __forceinline__ float2 div2_rn(float2 a, float2 nb, float2 r) {
    const float2 q0 = __fmul2_rn(a, r);
    const float2 rem = __ffma2_rd(q0, nb, a);
    return __ffma2_rn(rem, r, q0);
}

// ------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
    return v;
}

// Max over the aligned lane group of `lanes` (4 or 16) lanes.
template <int LANES>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int m = 1; m < LANES; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
    return v;
}

// Sum (or max, of values >= 0) over the `tpr` threads of one row. `part`
// holds one slot per warp of the CTA; warps of a row are contiguous. Every
// thread of the CTA must call it (it contains __syncthreads). Each warp of
// the row then reads the row's warp partials one per lane (at most 16, the
// rest 0) and combines them with the same xor butterfly, whose every step adds
// the same two operands in every lane: every thread of a row gets the
// bit-identical value, with no loop.
template <bool IS_MAX>
__device__ __forceinline__ float row_reduce(float v, float* part, int tpr, int lrow) {
    v = IS_MAX ? warp_max(v) : warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = v;
    __syncthreads();
    const int nw = tpr >> 5;
    const float r = lane < nw ? part[lrow * nw + lane] : 0.0f;
    return IS_MAX ? warp_max(r) : warp_sum(r);
}

// Sum of `a` and max of `b` (b >= 0) over the `tpr` threads of one row, in
// one shared-memory round (one __syncthreads); same rules as row_reduce.
// The max over a warp in one instruction (exact, as any order of maxima is).
__device__ __forceinline__ float warp_max_redux(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float2 row_reduce_sum_max(float a, float b, float2* part, int tpr, int lrow) {
    a = warp_sum(a);
    b = warp_max_redux(b);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = make_float2(a, b);
    __syncthreads();
    const int nw = tpr >> 5;
    const float2 r = lane < nw ? part[lrow * nw + lane] : make_float2(0.0f, 0.0f);
    return make_float2(warp_sum(r.x), warp_max_redux(r.y));
}

// ------------------------------------------------------------------ scales

// E8M0 code of an MX block: floor(log2(amax)) - 8 clamped to [-127, 127], plus
// the bias 127. For amax >= 2^-126 floor(log2(amax)) is the unbiased exponent
// field, so the code is that field minus 8; zero and subnormal amax (field 0)
// fall below -127 and clamp to code 0.
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
    const int field = (int)((__float_as_uint(amax) >> 23) & 0xFF);
    return (uint32_t)max(field - 8, 0);
}

// 2^-(code-127) = 2^(127-code) as a float; exact for every code in [0, 253].
__device__ __forceinline__ float mx_inv_scale(uint32_t code) {
    return __uint_as_float((254u - code) << 23);
}

}  // namespace sgq
