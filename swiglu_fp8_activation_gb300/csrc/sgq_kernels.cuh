// sgq_kernels.cuh -- the two row-engine kernels (add + RMSNorm, SwiGLU), each
// fused with FP8 quantisation in one of three formats. See sgq_device.cuh for
// the thread-to-data mapping.
#pragma once

#include "sgq_device.cuh"

namespace sgq {

struct NormArgs {
    const uint16_t* x;       // [M, H] bf16
    const uint16_t* r_in;    // [M, H] bf16 or null
    uint16_t* r_out;         // [M, H] bf16 or null (may equal r_in)
    const uint16_t* w;       // [H] bf16
    uint8_t* q;              // [M, H] E4M3
    void* scale;             // format-dependent scale array
    uint16_t* normed;        // [M, H] bf16 or null
    int64_t M;
    int H;
    int tpr;                 // threads per row (multiple of 32)
    int rpc;                 // rows per CTA
    float eps;
    uint32_t flags;
};

struct SwigluArgs {
    const uint16_t* gu;      // [M, 2I] bf16: gate = [0, I), up = [I, 2I)
    uint8_t* q;              // [M, I] E4M3
    void* scale;
    int64_t M;
    int I;
    int tpr;
    int rpc;
    uint32_t flags;
    int act;
    float alpha, beta, limit;
};

// Quantise the thread's NV chunks of one row (src = quant source values,
// zero in chunks past the row end or in rows past M) and store codes and
// scales. Every thread of the CTA must call it (the per-token format reduces
// over the row through shared memory).
//   MX:  code = E8M0 of the 1x32 block's amax; q = E4M3(src * 2^(127-code)),
//        the scaling being exact (a power of two).
//   FP8: s = amax / 448 (IEEE fp32 division); q = E4M3(src / s) with the IEEE
//        fp32 quotient (div_rn from one correctly rounded reciprocal per
//        group); s = 0 (all-zero group) stores s = 0 and q = 0.
template <int FMT, int NV>
__device__ __forceinline__ void quantize_store(const float (&src)[NV][8], int64_t row, bool row_ok,
                                               int t, int tpr, int lrow, int W, uint8_t* q,
                                               void* scale, float* part_amax) {
    const int nchunks = W >> 3;
    float row_amax = 0.0f;
    if (FMT == FMT_PT) {
        float m = 0.0f;
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(src[v][k]));
        row_amax = row_reduce<true>(m, part_amax, tpr, lrow);
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int c = t + v * tpr;
        float amax;
        if (FMT == FMT_PT) {
            amax = row_amax;
        } else {
            float m = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(src[v][k]));
            amax = group_max<FMT == FMT_MX ? 4 : 16>(m);   // all lanes take part
        }
        if (!row_ok || c >= nchunks) continue;
        float tq[8];
        if (FMT == FMT_MX) {
            const uint32_t code = mx_scale_code(amax);
            const float is = mx_inv_scale(code);
#pragma unroll
            for (int k = 0; k < 8; ++k) tq[k] = src[v][k] * is;
            if ((c & 3) == 0) static_cast<uint8_t*>(scale)[row * (W >> 5) + (c >> 2)] = (uint8_t)code;
        } else {
            const float s = __fdiv_rn(amax, 448.0f);
            if (s >= 0x1p-126f) {
                const float r = __frcp_rn(s);   // once per group, then one FMA pair per element
#pragma unroll
                for (int k = 0; k < 8; ++k) tq[k] = div_rn(src[v][k], s, r);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) tq[k] = (s == 0.0f) ? 0.0f : __fdiv_rn(src[v][k], s);
            }
            if (FMT == FMT_B128 && (c & 15) == 0) static_cast<float*>(scale)[row * (W >> 7) + (c >> 4)] = s;
            if (FMT == FMT_PT && c == 0) static_cast<float*>(scale)[row] = s;
        }
        const uint2 packed = make_uint2(f32x4_to_e4m3x4(tq[0], tq[1], tq[2], tq[3]),
                                        f32x4_to_e4m3x4(tq[4], tq[5], tq[6], tq[7]));
        st8(q + row * W + (int64_t)c * 8, packed);
    }
}

// Residual add + RMSNorm + quantisation. One row per `tpr` threads.
template <int FMT, int NV>
__global__ void __launch_bounds__(kMaxTPR) norm_quant_kernel(const NormArgs a) {
    __shared__ float part_ss[32];
    __shared__ float part_amax[32];
    const int tpr = a.tpr;
    const int lrow = threadIdx.x / tpr;
    const int t = threadIdx.x - lrow * tpr;
    const int64_t row = (int64_t)blockIdx.x * a.rpc + lrow;
    const bool row_ok = row < a.M;
    const int H = a.H, nchunks = H >> 3;
    const int64_t base = row * (int64_t)H;

    // 1. issue every load of the row (x, r and the weight) before any arithmetic
    pdl_wait();
    uint4 xv[NV], rv[NV], wv[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int c = t + v * tpr;
        const bool ok = row_ok && c < nchunks;
        xv[v] = ok ? ld_once(a.x + base + (int64_t)c * 8) : make_uint4(0, 0, 0, 0);
        rv[v] = (ok && a.r_in) ? ld_coherent(a.r_in + base + (int64_t)c * 8) : make_uint4(0, 0, 0, 0);
        wv[v] = ok ? ld_shared_by_rows(a.w + (int64_t)c * 8) : make_uint4(0, 0, 0, 0);
    }
    pdl_trigger();

    // 2. h = x + r in fp32; write the updated residual; partial sum of squares
    float h[NV][8];
    float ss = 0.0f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int c = t + v * tpr;
        bf16x8_to_f32(xv[v], h[v]);
        if (a.r_in) {
            float rf[8];
            bf16x8_to_f32(rv[v], rf);
#pragma unroll
            for (int k = 0; k < 8; ++k) h[v][k] += rf[k];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) ss = fmaf(h[v][k], h[v][k], ss);
        if (a.r_out && row_ok && c < nchunks) st16(a.r_out + base + (int64_t)c * 8, f32x8_to_bf16x8(h[v]));
    }

    // 3. inv = 1/sqrt(mean(h^2) + eps), each step correctly rounded
    ss = row_reduce<false>(ss, part_ss, tpr, lrow);
    const float inv = __frsqrt_rn(__fdiv_rn(ss, (float)H) + a.eps);

    // 4. y = h * inv * (1 + w) or h * inv * w; bf16 copy; quant source
    const bool gemma = (a.flags & F_GEMMA) != 0, from32 = (a.flags & F_FROM_FP32) != 0;
    float src[NV][8];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int c = t + v * tpr;
        if (!(row_ok && c < nchunks)) {
#pragma unroll
            for (int k = 0; k < 8; ++k) src[v][k] = 0.0f;
            continue;
        }
        float wf[8], y[8];
        bf16x8_to_f32(wv[v], wf);
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = h[v][k] * inv * (gemma ? 1.0f + wf[k] : wf[k]);
        const uint4 yb = f32x8_to_bf16x8(y);
        if (a.normed) st16(a.normed + base + (int64_t)c * 8, yb);
        if (from32) {
#pragma unroll
            for (int k = 0; k < 8; ++k) src[v][k] = y[k];
        } else {
            bf16x8_to_f32(yb, src[v]);
        }
    }

    // 5. group amax, scales, E4M3 codes
    quantize_store<FMT, NV>(src, row, row_ok, t, tpr, lrow, H, a.q, a.scale, part_amax);
}

// The activation of two (gate, up) pairs, in fp32:
//   OAI:  g' = min(g, limit), u' = min(max(u, -limit), limit),
//         a = (g' * sigmoid(alpha * g')) * (u' + beta); alpha * g' is carried
//         with its exact FMA residual into the sigmoid;
//   SiLU: a = (g * sigmoid(g)) * u, the first factor rounded to bf16 when
//         round_silu is set.
template <int ACT>
__device__ __forceinline__ float2 activation2(float2 g, float2 u, float alpha, float beta, float limit,
                                              bool round_silu) {
    if (ACT == ACT_OAI) {
        const float2 gc = make_float2(fminf(g.x, limit), fminf(g.y, limit));
        const float2 uc = make_float2(fminf(fmaxf(u.x, -limit), limit), fminf(fmaxf(u.y, -limit), limit));
        const float2 zh = __fmul2_rn(f2(alpha), gc);
        const float2 zl = __ffma2_rn(f2(alpha), gc, __fmul2_rn(zh, f2(-1.0f)));
        return __fmul2_rn(__fmul2_rn(gc, sigmoid2(zh, zl)), __fadd2_rn(uc, f2(beta)));
    }
    float2 s = __fmul2_rn(g, sigmoid2(g, f2(0.0f)));
    if (round_silu) s = make_float2(round_bf16(s.x), round_bf16(s.y));
    return __fmul2_rn(s, u);
}

// SwiGLU + quantisation. One row per `tpr` threads.
template <int FMT, int NV, int ACT>
__global__ void __launch_bounds__(kMaxTPR) swiglu_quant_kernel(const SwigluArgs a) {
    __shared__ float part_amax[32];
    const int tpr = a.tpr;
    const int lrow = threadIdx.x / tpr;
    const int t = threadIdx.x - lrow * tpr;
    const int64_t row = (int64_t)blockIdx.x * a.rpc + lrow;
    const bool row_ok = row < a.M;
    const int I = a.I, nchunks = I >> 3;
    const uint16_t* grow = a.gu + row * (int64_t)(2 * I);

    pdl_wait();
    uint4 gv[NV], uv[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int c = t + v * tpr;
        const bool ok = row_ok && c < nchunks;
        gv[v] = ok ? ld_once(grow + (int64_t)c * 8) : make_uint4(0, 0, 0, 0);
        uv[v] = ok ? ld_once(grow + I + (int64_t)c * 8) : make_uint4(0, 0, 0, 0);
    }
    pdl_trigger();

    const bool round_silu = (a.flags & F_ACT_BF16) != 0;
    float src[NV][8];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        float g[8], u[8];
        bf16x8_to_f32(gv[v], g);
        bf16x8_to_f32(uv[v], u);
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float2 act = activation2<ACT>(make_float2(g[k], g[k + 1]), make_float2(u[k], u[k + 1]),
                                                a.alpha, a.beta, a.limit, round_silu);
            src[v][k] = act.x;
            src[v][k + 1] = act.y;
        }
    }
    if (!(a.flags & F_FROM_FP32)) {    // quantise the bf16 rounding of the activation
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int k = 0; k < 8; ++k) src[v][k] = round_bf16(src[v][k]);
    }
    // chunks past the row end loaded zeros, and every activation of 0 and 0 is 0

    quantize_store<FMT, NV>(src, row, row_ok, t, tpr, lrow, I, a.q, a.scale, part_amax);
}

}  // namespace sgq
