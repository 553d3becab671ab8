// sgq_device.cuh -- device code of the fused norm / SwiGLU + FP8 quantisation
// kernels for sm_103a.
//
// One "row engine" serves both operations. A row of W elements is split into
// 16-byte chunks of 8 bf16 values; `tpr` threads (a multiple of 32) own one
// row, and thread t owns chunks t, t + tpr, ..., t + (NV-1)*tpr, so every
// warp-wide load is 512 contiguous bytes. All NV chunks of a thread are loaded
// before any arithmetic (the whole row sits in registers: no second read of
// global memory and no shared-memory staging of the row). Reductions:
//   * sum of squares (RMSNorm) and per-token amax: warp shuffles, then one
//     shared-memory step across the row's warps;
//   * 1x32 (MX) amax: the 4 lanes that own one 32-block (2 xor-shuffles);
//   * 1x128 amax: the 16 lanes that own one 128-block (4 xor-shuffles).
// Block alignment holds because tpr is a multiple of 32 and W is a multiple
// of the group size: chunk c lives in lane c % 32 of its warp, so a 32-block
// (4 chunks) or a 128-block (16 chunks) never straddles a lane group.
//
// Numeric formats: bf16 = upper half of IEEE binary32; E4M3 = OCP "e4m3fn";
// E8M0 = OCP MX scale byte, value 2^(code-127). The operations follow
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

constexpr uint32_t F_GEMMA = 1u << 0;
constexpr uint32_t F_FROM_FP32 = 1u << 1;
constexpr uint32_t F_ACT_BF16 = 1u << 2;

constexpr int kMaxNV = 4;          // chunks per thread
constexpr int kMaxTPR = 512;       // threads per row (SGQ_MAX_WIDTH = kMaxTPR * kMaxNV * 8)
constexpr int kTargetCTA = 256;    // threads per CTA when several rows share one

// ----------------------------------------------------------------- memory

// Streaming 16-byte load of data read once by this kernel (x, gate_up):
// non-coherent path, no L1 allocation, 256-byte L2 prefetch.
__device__ __forceinline__ uint4 ld_once(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte load through the coherent path (the residual may be updated in place).
__device__ __forceinline__ uint4 ld_coherent(const void* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte load of data every row reads (the norm weight): cached.
__device__ __forceinline__ uint4 ld_shared_by_rows(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void st16(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st8(void* p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
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

// Round a float to the nearest bf16 (ties to even) and widen it back.
__device__ __forceinline__ float round_bf16(float v) {
    return __uint_as_float(f32x2_to_bf16x2(v, 0.0f) << 16);
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
// before its first global memory access, so an early start is always safe.
// pdl_trigger() lets the next grid on the stream begin launching; that grid
// in turn waits in its own pdl_wait() before touching memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------ arithmetic

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(e) split into an fp32 head (round to nearest) and the fp32 rounding of
// the remainder.
constexpr float kLog2eHi = 1.44269502162933349609375f;   // 0x3FB8AA3B
constexpr float kLog2eLo = 1.925963033500011e-08f;       // log2(e) - kLog2eHi
// 1.5 * 2^23: adding it to |x| < 2^22 rounds x to an integer (to nearest even)
// held in the low mantissa bits.
constexpr float kRoundMagic = 12582912.0f;

// 2^x for |x| <= 0.5005: degree-6 polynomial whose coefficients were fitted
// for least relative error (Lawson-weighted least squares on 4000 Chebyshev
// nodes, then rounded to fp32). Fit error 1.9e-9; fp32 Horner evaluation
// stays within 1.4 ulp.
constexpr float kExp2C0 = 1.0f, kExp2C1 = 0.6931471824645996f, kExp2C2 = 0.24022646248340607f,
                kExp2C3 = 0.05550328269600868f, kExp2C4 = 0.009618490003049374f,
                kExp2C5 = 0.0013400063617154956f, kExp2C6 = 0.00015345696010626853f;

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// Logistic sigmoid 1/(1 + e^-z) of two values, z = zh + zl (zl: the exact
// residual of the fp32 product that formed zh, or 0). Written from the
// mathematics, on packed fp32x2 arithmetic, with every term kept on the
// negative side so that no operand needs a separate negation:
//   * E = e^-|z| = 2^q, q = -|z| log2 e carried as head qh = RN(-|z| log2e_hi)
//     plus tail (the FMA residual of that product, |z| log2e_lo and the
//     residual zl), in the manner of Cody and Waite's argument reduction;
//   * q = n + f with n = round(qh) <= 0 and |f| <= 0.5005: 2^f from the
//     polynomial above, times 2^n by adding n to the exponent field (two
//     steps when E falls below the normal range, a rare branch);
//   * sigmoid(|z|) = 1/(1+E) and sigmoid(-|z|) = E/(1+E), the hardware
//     reciprocal refined by one Newton-Raphson step.
// |z| is capped at 128, where e^-128 underflows fp32. Relative error about
// 2 ulp.
__device__ __forceinline__ float2 sigmoid2(float2 zh, float2 zl) {
    const float2 az = make_float2(fminf(fabsf(zh.x), 128.0f), fminf(fabsf(zh.y), 128.0f));
    // |z| = az + azl: the residual takes the sign of zh (it is zero past the cap)
    const float2 azl = make_float2(
        fabsf(zh.x) <= 128.0f ? __uint_as_float(__float_as_uint(zl.x) ^ (__float_as_uint(zh.x) & 0x80000000u)) : 0.0f,
        fabsf(zh.y) <= 128.0f ? __uint_as_float(__float_as_uint(zl.y) ^ (__float_as_uint(zh.y) & 0x80000000u)) : 0.0f);
    const float2 qh = __fmul2_rn(az, f2(-kLog2eHi));                     // -|z| log2e, rounded
    float2 tail = __ffma2_rn(az, f2(kLog2eHi), qh);                      // |z| log2e_hi + qh, exact
    tail = __ffma2_rn(az, f2(kLog2eLo), tail);
    tail = __ffma2_rn(azl, f2(kLog2eHi), tail);                          // q = qh - tail
    const float2 big = __fadd2_rn(qh, f2(kRoundMagic));                  // round(qh) in the low bits
    const float2 n = __fadd2_rn(big, f2(-kRoundMagic));
    float2 f = __ffma2_rn(n, f2(-1.0f), qh);                             // qh - n, exact
    f = __ffma2_rn(tail, f2(-1.0f), f);
    float2 e = __ffma2_rn(f2(kExp2C6), f, f2(kExp2C5));
    e = __ffma2_rn(e, f, f2(kExp2C4));
    e = __ffma2_rn(e, f, f2(kExp2C3));
    e = __ffma2_rn(e, f, f2(kExp2C2));
    e = __ffma2_rn(e, f, f2(kExp2C1));
    e = __ffma2_rn(e, f, f2(kExp2C0));                                   // 2^f in [0.7, 1.42]
    // 2^n: add n to the exponent field. Exact while n >= -125 (e's field is 126 or 127).
    const int nx = __float_as_int(big.x) - __float_as_int(kRoundMagic);
    const int ny = __float_as_int(big.y) - __float_as_int(kRoundMagic);
    if (min(nx, ny) >= -125) {
        e = make_float2(__uint_as_float(__float_as_uint(e.x) + ((uint32_t)nx << 23)),
                        __uint_as_float(__float_as_uint(e.y) + ((uint32_t)ny << 23)));
    } else {   // |z| > 86.6: E below the normal range, scale in two exact steps
        e = make_float2(__uint_as_float(__float_as_uint(e.x) + ((uint32_t)max(nx, -125) << 23)),
                        __uint_as_float(__float_as_uint(e.y) + ((uint32_t)max(ny, -125) << 23)));
        e = __fmul2_rn(e, make_float2(__uint_as_float((uint32_t)(127 + min(nx + 125, 0)) << 23),
                                      __uint_as_float((uint32_t)(127 + min(ny + 125, 0)) << 23)));
    }
    const float2 d = __fadd2_rn(e, f2(1.0f));
    const float2 nd = __ffma2_rn(e, f2(-1.0f), f2(-1.0f));               // -(1 + E)
    const float2 r0 = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    const float2 res = __ffma2_rn(nd, r0, f2(1.0f));                     // 1 - d*r0
    const float2 r = __ffma2_rn(r0, res, r0);                            // one Newton-Raphson step
    const float2 er = __fmul2_rn(e, r);
    return make_float2(zh.x < 0.0f ? er.x : r.x, zh.y < 0.0f ? er.y : r.y);
}

// a / b rounded to nearest even, given r = RN(1/b) (b and r normal). q0 = a*r
// is within one ulp of a/b; the remainder a - b*q0 is exact in one FMA, and
// q0 + rem*r rounded once is the correctly rounded quotient (Markstein's
// correction step: P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990). Results
// below the normal range may differ from IEEE division by an ulp.
__device__ __forceinline__ float div_rn(float a, float b, float r) {
    const float q0 = a * r;
    const float rem = fmaf(-q0, b, a);
    return fmaf(rem, r, q0);
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

// Sum (or max) over the `tpr` threads of one row. `part` holds one slot per
// warp of the CTA; warps of a row are contiguous. Every thread of the CTA must
// call it (it contains __syncthreads). The row's warp partials are combined in
// warp order, so every thread of a row gets the same value.
template <bool IS_MAX>
__device__ __forceinline__ float row_reduce(float v, float* part, int tpr, int lrow) {
    v = IS_MAX ? warp_max(v) : warp_sum(v);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) part[warp] = v;
    __syncthreads();
    const int w0 = lrow * (tpr >> 5), nw = tpr >> 5;
    float r = part[w0];
    for (int i = 1; i < nw; ++i) r = IS_MAX ? fmaxf(r, part[w0 + i]) : r + part[w0 + i];
    return r;
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
