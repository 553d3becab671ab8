// sgq_kernels.cuh -- the row-engine kernels: add + RMSNorm (one row set, or
// two in one launch) and SwiGLU, each fused with FP8 quantisation in one of
// three formats, and the standalone quantisation of the unfused chains. See
// sgq_device.cuh for the thread-to-data mapping.
#pragma once

#include <type_traits>

#include "sgq_device.cuh"

namespace sgq {

// Where a kernel writes its scales. Scales of group g of row `row` go to
// base(row) + (g / 4) * s4 + (g % 4) * s1 bytes (scale_row), which covers:
//   SCALE_ROW_MAJOR  [M, ng] row-major;
//   SCALE_SWIZZLED   MXFP8 E8M0 in 128 x 4 tiles of 512 bytes, tiles row-major
//                    over (M/128 bands) x (ng/4 tile columns); inside a tile,
//                    row r and column j at (r % 32) * 16 + (r / 32) * 4 + j;
//   SCALE_COL_MAJOR  fp32 [ng, ld] (group-major), ld = M rounded up to 4.
// Rows in [M, Ms) are padding of the layout: their scales are written as
// zero (their inputs read as zero), and nothing else of them is written.
struct ScaleOut {
    void* p;
    int64_t ld;       // SCALE_SWIZZLED: tiles per 128-row band; SCALE_COL_MAJOR: leading dimension
    int64_t Ms;       // rows whose scales are written (M, or M padded to the layout's row multiple)
    int ng;           // groups per row
    int layout;       // SCALE_*
};

struct NormArgs {
    const uint16_t* x;       // [M, ldx] 16-bit (bf16 or fp16), rows read from column 0 to H
    const uint16_t* r_in;    // [M, H] bf16 or null
    uint16_t* r_out;         // [M, H] bf16 or null (may equal r_in)
    const uint16_t* w;       // [H] bf16
    uint8_t* q;              // [M, H] E4M3, or null (no quantisation)
    ScaleOut so;
    uint16_t* normed;        // [M, H] bf16 or null
    int64_t M;
    int64_t ldx;             // row stride of x in elements (H for contiguous rows)
    int H;
    int tpr;                 // threads per row (multiple of 32)
    int rpc;                 // rows per CTA
    float eps;
    uint32_t flags;
    int segc;                // output chunks a column segment (SEG) or cluster CTA (CL); H / 8 for whole rows
};

// The all-reduce norm's partial inputs: the tensor-parallel ranks' [M, H]
// rows, summed into x (NormArgs::x is then unused). A parameter of that
// kernel alone, so the other norms' launches carry none of it.
struct ARParts {
    int n;
    const uint16_t* p[kMaxRanks];
};

struct NormARArgs {
    NormArgs a;
    ARParts ar;
};

struct SwigluArgs {
    const uint16_t* gu;      // [M, 2I] bf16: gate = [0, I), up = [I, 2I)
    uint8_t* q;              // [M, I] E4M3 (null when `out` is set)
    ScaleOut so;
    uint16_t* out;           // [M, I] bf16 activation instead of quantising, or null
    int64_t M;
    int I;
    int tpr;
    int rpc;
    uint32_t flags;
    int act;
    float alpha, beta, limit;
    uint32_t lim2, nlim2;    // bf16x2 of limit and -limit (the CLAMP16 kernels)
    uint32_t tail2;          // bf16x2 of the least gate t with RN(khi t) <= 125 (the CLAMP16 kernels)
    float khi, klo;          // -alpha log2(e) in two fp32 parts (OAI)
    int segc;                // chunks a column segment or cluster CTA (I / 8 when rows are whole)
};

struct QuantArgs {
    const uint16_t* src;     // [M, W] bf16 or fp16
    uint8_t* q;              // [M, W] E4M3
    ScaleOut so;
    int64_t M;
    int W;
    int tpr;
    int rpc;
    int segc;                // chunks a column segment or cluster CTA (W / 8 when rows are whole)
};

// One row's view of ScaleOut in layout LAYOUT (a compile-time choice, so
// that each layout's address arithmetic is only what it needs).
struct ScaleRow {
    char* base;       // byte address of group 0 of the row
    int64_t ld4;      // SCALE_COL_MAJOR: bytes from one group's column to the next
    int pad_last;     // SCALE_SWIZZLED with ng % 4 != 0: the last real group, whose
                      // tile row is completed with zero codes; else -1
};

template <int FMT, int LAYOUT>
__device__ __forceinline__ ScaleRow scale_row(const ScaleOut& so, int64_t row) {
    char* p = static_cast<char*>(so.p);
    ScaleRow r;
    r.ld4 = 0;
    r.pad_last = -1;
    if (FMT == FMT_PT) {
        r.base = p + row * 4;
    } else if (LAYOUT == SCALE_SWIZZLED) {
        r.base = p + (row >> 7) * so.ld * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
        if (so.ng & 3) r.pad_last = so.ng - 1;
    } else if (LAYOUT == SCALE_COL_MAJOR) {
        r.base = p + row * 4;
        r.ld4 = so.ld * 4;
    } else {
        r.base = p + row * (int64_t)so.ng * (FMT == FMT_MX ? 1 : 4);
    }
    return r;
}

// Byte address of group g's scale in the row.
template <int FMT, int LAYOUT>
__device__ __forceinline__ char* scale_addr(const ScaleRow& r, int g) {
    if (LAYOUT == SCALE_SWIZZLED) return r.base + ((g >> 2) << 9) + (g & 3);
    if (LAYOUT == SCALE_COL_MAJOR) return r.base + g * r.ld4;
    return r.base + g * (FMT == FMT_MX ? 1 : 4);
}

// The FP8 scale amax / 448, correctly rounded: the Markstein quotient with
// RN(1/448) where the quotient is normal, IEEE division below.
__device__ __forceinline__ float fp8_scale(float amax) {
    return amax >= 0x1p-100f ? div_rn(amax, 448.0f, kInv448) : __fdiv_rn(amax, 448.0f);
}

// Quantise one chunk (8 source values of row `row`, chunk index c) and store
// its 8 E4M3 codes and, from the first chunk of its group, the scale. Every
// lane of the warp must call it for MX and 1x128 (the group amax is a lane
// shuffle); `store` is false for lanes without a valid chunk (their src is 0)
// and `sstore` likewise for the scale (true also on the layout's padding rows).
//   MX:  code = E8M0 of the 1x32 block's amax; q = E4M3(src * 2^(127-code)),
//        the scaling being exact (a power of two).
//   FP8: s = amax / 448 (IEEE fp32 division); q = E4M3(src / s) with the IEEE
//        fp32 quotient (div_rn from one correctly rounded reciprocal per
//        group); s = 0 (all-zero group) stores s = 0 and q = 0. The per-token
//        format passes its row scale and reciprocal in (pt_s, pt_r).
template <int FMT, int LAYOUT>
__device__ __forceinline__ void quantize_chunk(const float (&src)[8], int64_t row, int c, bool store, bool sstore,
                                               int W, uint8_t* q, const ScaleRow& sr, float pt_s = 0.0f,
                                               float pt_r = 0.0f) {
    float m = 0.0f;
    if (FMT != FMT_PT) {
#pragma unroll
        for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(src[k]));
        m = group_max<FMT == FMT_MX ? 4 : 16>(m);        // all lanes take part
    }
    float tq[8];
    if (FMT == FMT_MX) {
        const uint32_t code = mx_scale_code(m);
        const float is = mx_inv_scale(code);
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float2 t = __fmul2_rn(make_float2(src[k], src[k + 1]), f2(is));
            tq[k] = t.x;
            tq[k + 1] = t.y;
        }
        const int g = c >> 2;
        uint8_t* sp = reinterpret_cast<uint8_t*>(scale_addr<FMT, LAYOUT>(sr, g));
        const bool lead = sstore && (c & 3) == 0;
        st_u8_if(sp, code, lead);
        if (LAYOUT == SCALE_SWIZZLED && g == sr.pad_last && lead) {   // zero codes complete the last tile row
            for (int j = (g & 3) + 1; j < 4; ++j) sp[j - (g & 3)] = 0;
        }
    } else {
        float s = pt_s, r = pt_r;
        if (FMT == FMT_B128) {
            s = fp8_scale(m);
            r = s >= 0x1p-126f ? __frcp_rn(s) : 0.0f;   // once per group
        }
        if (s >= 0x1p-126f || s == 0.0f) {              // r = 0 for s = 0: every code is 0
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                const float2 t = div2_rn(make_float2(src[k], src[k + 1]), f2(-s), f2(r));
                tq[k] = t.x;
                tq[k + 1] = t.y;
            }
        } else {                                         // subnormal scale (amax < 5.3e-36)
#pragma unroll
            for (int k = 0; k < 8; ++k) tq[k] = __fdiv_rn(src[k], s);
        }
        if (FMT == FMT_B128) {
            const int g = c >> 4;
            st_f32_if(reinterpret_cast<float*>(scale_addr<FMT, LAYOUT>(sr, g)), s, sstore && (c & 15) == 0);
        } else {
            st_f32_if(reinterpret_cast<float*>(sr.base), s, sstore && c == 0);
        }
    }
    const uint2 packed = make_uint2(f32x4_to_e4m3x4(tq[0], tq[1], tq[2], tq[3]),
                                    f32x4_to_e4m3x4(tq[4], tq[5], tq[6], tq[7]));
    st8_if(q + row * W + (int64_t)c * 8, packed, store);
}

// Per-token scale and its reciprocal from the row amax (one per row).
__device__ __forceinline__ float2 per_token_scale(float row_amax) {
    const float s = fp8_scale(row_amax);
    return make_float2(s, s >= 0x1p-126f ? __frcp_rn(s) : 0.0f);
}

// Residual add + RMSNorm + quantisation. One row per `tpr` threads.
// y is formed as inv * (h * w'), w' = 1 + w or w: the per-token format then
// needs no second reduction, since inv > 0 and rounding is monotone, so
// RN(inv * max|h w'|) is exactly the largest |y| (and its bf16 rounding the
// largest bf16 |y|); the max of |h w'| travels with the sum of squares.
// Inputs staged per chunk by the norm kernel: x, the residual (if any) and w.
__host__ __device__ constexpr int norm_stage_inputs(bool has_res) { return has_res ? 3 : 2; }
__host__ __device__ constexpr int norm_stage_bytes(bool has_res, int nv, int threads) {
    return nv * norm_stage_inputs(has_res) * threads * 16;
}

// The rows of CTA `blk` of one norm launch (blockDim.x = a.rpc * a.tpr).
// FULL: every thread's chunks lie inside the row and every row inside M (the
// plan divides both exactly), so no bounds are checked. DT is the 16-bit
// type of x, r, w and the written rows.
// SEG: column segments (the bounds-checked single norm): each row may run as
// gridDim.y CTAs. Every one of them reads the whole row of x and r and forms
// the same sum of squares (and max |z|) in the same order, so all get the
// bit-identical inv; CTA y then writes only chunks [y * segc, (y + 1) * segc),
// segc a multiple of 32, so that a warp's chunks are all in or all out. The
// host never splits an in-place residual update, which another CTA of the row
// would read back.
// AR: x is the all-reduce of ar->n partial inputs (the tensor-parallel
// ranks' [M, H] rows): their sum in fp32, in rank order, rounded once to the
// activation type, as an all-reduce's output would be; each partial is
// staged in a shared-memory slot of its own beside r and w.
// CL: a row wider than one CTA covers, split over the CTAs of a cluster (one
// row per cluster, blk = the row): CTA k of the cluster reads, computes and
// writes only chunks [k * segc, min((k + 1) * segc, H / 8)), segc a multiple
// of 32, and the CTAs' partial sums of squares (and max |z|) are combined in
// rank order through shared memory (cluster_combine), so every CTA of the row
// gets the bit-identical inv. Each CTA reads only its own columns, so an
// in-place residual update is safe here too.
template <int FMT, int LAYOUT, int NV, bool HAS_RES, bool FULL, int DT, bool SEG = false, bool CL = false,
          bool AR = false>
__device__ __forceinline__ void norm_rows(const NormArgs& a, int64_t blk, const ARParts* ar = nullptr) {
    extern __shared__ uint4 stage[];
    __shared__ float2 part[32];
    constexpr int NIN = norm_stage_inputs(HAS_RES);
    // shared-memory slots a chunk: x (AR: one for each partial), r, w
    const int nparts = AR ? ar->n : 1;
    const int nslot = AR ? nparts + NIN - 1 : NIN;
    const int ir = AR ? nparts : 1, iw = nslot - 1;
    const int tpr = a.tpr;
    const int nt = blockDim.x;
    // one row a CTA (the per-token format's wide rows): no division
    const int lrow = (FMT == FMT_PT && a.rpc == 1) ? 0 : threadIdx.x / tpr;
    const int t = threadIdx.x - lrow * tpr;
    const int64_t row = blk * a.rpc + lrow;
    const bool row_ok = FULL || row < a.M;
    const int H = a.H, nchunks = H >> 3;
    const int64_t base = row * (int64_t)H;
    auto slot = [&](int v, int i) { return &stage[(nslot * v + i) * nt + threadIdx.x]; };
    const int cb = SEG ? (int)blockIdx.y * a.segc : CL ? (int)cluster_rank() * a.segc : 0;   // the chunks this CTA writes
    const int cend = SEG ? cb + a.segc : CL ? min(cb + a.segc, nchunks) : nchunks;
    const int c0 = CL ? cb : 0;              // chunk of thread 0's first copy (CL: the segment's first)
    const int clim = CL ? cend : nchunks;    // chunks this CTA reads end here

    // 1. every load of the row (x, r and the weight) goes out at once, copied
    //    asynchronously into this thread's shared-memory slots. The weight is
    //    not written by the grid this launch may overlap (a contract of the
    //    entry points), so its copies go out before pdl_wait() as one commit
    //    group of their own; then x and r, one commit group per chunk. A
    //    thread reads back only its own slots, and writes the updated residual
    //    of a chunk only after that chunk's group has landed, so an in-place
    //    residual update is safe.
    // SEG: the weight only where this CTA writes (the per-token max |z| needs all of it)
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int c = c0 + t + v * tpr;
        const bool okw = (FULL || (row_ok && c < clim)) && (!SEG || FMT == FMT_PT || (c >= cb && c < cend));
        cp_async16_cached(slot(v, iw), okw ? (const void*)(a.w + (int64_t)c * 8) : (const void*)a.w, okw ? 16 : 0);
    }
    cp_async_commit();
    pdl_wait();
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int c = c0 + t + v * tpr;
        const bool ok = FULL || (row_ok && c < clim);      // else zero-fill, reading nothing
        const int nb = ok ? 16 : 0;
        if (AR) {
            for (int p = 0; p < nparts; ++p)
                cp_async16(slot(v, p), ok ? (const void*)(ar->p[p] + base + (int64_t)c * 8) : (const void*)a.w, nb);
        } else {
            cp_async16(slot(v, 0), ok ? (const void*)(a.x + row * a.ldx + (int64_t)c * 8) : (const void*)a.x, nb);
        }
        if (HAS_RES)
            cp_async16(slot(v, ir), ok ? (const void*)(a.r_in + base + (int64_t)c * 8) : (const void*)a.w, nb);
        cp_async_commit();
    }
    pdl_trigger();
    if (CL) cluster_arrive_relaxed();       // completed in cluster_combine, once the whole cluster runs

    // 2. h = x + r in fp32; write the updated residual; z = h * w'; partial
    //    sum of squares (and max |z| for the per-token format). SEG: warps
    //    whose chunks lie outside this CTA's segment only add their h^2 to the
    //    sum (c & ~31 is the same in every lane of a warp, and segc is a
    //    multiple of 32); their z is never used, except by the per-token max.
    const bool from32 = (a.flags & F_FROM_FP32) != 0;
    float z[NV][8];
    float2 ss2 = make_float2(0.0f, 0.0f);
    float zmax = 0.0f;
    // The weight term w' = w + 1 (Gemma) or w + (-0), which is w exactly,
    // signed zeros included: an addition of w_add in the general form
    // (WMODE 0); the per-token kernels take the weight form as a constant
    // (WMODE 1: + 1, WMODE 2: no addition), the same values. (For every
    // format, the doubled code measured 10% slower at small M.)
    const float w_add = (a.flags & F_GEMMA) ? 1.0f : -0.0f;
    auto pass1 = [&](auto wmode_tag) {
        constexpr int WMODE = decltype(wmode_tag)::value;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int c = c0 + t + v * tpr;
            const bool mine = !SEG || FMT == FMT_PT || ((c & ~31) >= cb && (c & ~31) < cend);
            float h[8], wf[8];
            cp_async_wait_group_of<NV>(v);
            load8<DT>(ld_smem16(slot(v, 0)), h);
            if (AR) {                        // x = the partials' sum in rank order, rounded to DT
                for (int p = 1; p < nparts; ++p) {
                    float pf[8];
                    load8<DT>(ld_smem16(slot(v, p)), pf);
#pragma unroll
                    for (int k = 0; k < 8; k += 2) {
                        const float2 hs = __fadd2_rn(make_float2(h[k], h[k + 1]), make_float2(pf[k], pf[k + 1]));
                        h[k] = hs.x;
                        h[k + 1] = hs.y;
                    }
                }
                load8<DT>(pack8<DT>(h), h);
            }
            if (HAS_RES) {
                float rf[8];
                load8<DT>(ld_smem16(slot(v, ir)), rf);
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    const float2 hs = __fadd2_rn(make_float2(h[k], h[k + 1]), make_float2(rf[k], rf[k + 1]));
                    h[k] = hs.x;
                    h[k + 1] = hs.y;
                }
                // the updated residual is next read by the following layer's norm,
                // after the sublayer in between: streamed out (evict-first)
                if (a.r_out && mine)
                    st16_cs_if(a.r_out + base + (int64_t)c * 8, pack8<DT>(h),
                               FULL || (row_ok && (SEG ? c >= cb && c < cend : c < clim)));
            }
            if (!mine) {
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    const float2 hp = make_float2(h[k], h[k + 1]);
                    ss2 = __ffma2_rn(hp, hp, ss2);
                }
                continue;
            }
            load8<DT>(ld_smem16(slot(v, iw)), wf);
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                const float2 hp = make_float2(h[k], h[k + 1]);
                float2 wp = make_float2(wf[k], wf[k + 1]);
                if constexpr (WMODE == 0) wp = __fadd2_rn(wp, f2(w_add));
                else if constexpr (WMODE == 1) wp = __fadd2_rn(wp, f2(1.0f));
                ss2 = __ffma2_rn(hp, hp, ss2);
                const float2 zp = __fmul2_rn(hp, wp);
                z[v][k] = zp.x;
                z[v][k + 1] = zp.y;
                if (FMT == FMT_PT) zmax = fmaxf(zmax, fmaxf(fabsf(zp.x), fabsf(zp.y)));
            }
        }
    };
    if constexpr (FMT == FMT_PT) {
        if (a.flags & F_GEMMA) pass1(std::integral_constant<int, 1>{});
        else pass1(std::integral_constant<int, 2>{});
    } else {
        pass1(std::integral_constant<int, 0>{});
    }
    float ss = ss2.x + ss2.y;

    // 3. inv = 1/sqrt(mean(h^2) + eps), each step correctly rounded
    float row_zmax = 0.0f;
    if (FMT == FMT_PT) {
        const float2 r = row_reduce_sum_max(ss, zmax, part, tpr, lrow);
        ss = r.x;
        row_zmax = r.y;
    } else {
        ss = row_reduce<false>(ss, reinterpret_cast<float*>(part), tpr, lrow);
    }
    if (CL) {                                // the row's totals over the cluster, in rank order
        __shared__ float2 cl_slots[kMaxCluster];
        const float2 r = cluster_combine(make_float2(ss, row_zmax), cl_slots);
        ss = r.x;
        row_zmax = r.y;
    }
    float inv = __frsqrt_rn(__fdiv_rn(ss, (float)H) + a.eps);
    if (!FULL && !row_ok) inv = 0.0f;                          // a padding row of the scale layout: all zero

    // 4. y = inv * z; 16-bit copy; quant source; quantise (MX and 1x128 chunk by
    //    chunk; per-token after the whole row, with the row scale from ymax).
    //    Without q (the unfused norm) only the bf16 copy is written.
    const bool quant = a.q != nullptr;
    const bool srow_ok = FULL || row < a.so.Ms;
    const ScaleRow sr = scale_row<FMT, LAYOUT>(a.so, row);
    float2 pt = make_float2(0.0f, 0.0f);
    if (FMT == FMT_PT) {
        const float ymax = inv * row_zmax;                     // = max |y| exactly
        pt = per_token_scale(from32 ? ymax : round_io<DT>(ymax));
    }
    const bool normed = a.normed != nullptr;
    // the chunk loop, specialised for the three cases (no quantisation; a
    // 16-bit or an fp32 quant source) so that no per-chunk branch remains
    auto emit = [&](auto quant_tag, auto from32_tag) {
        constexpr bool QUANT = decltype(quant_tag)::value, FROM32 = decltype(from32_tag)::value;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int c = c0 + t + v * tpr;
            // warps whose chunks lie outside this CTA's segment (or wholly past
            // the row end) skip the chunk; c & ~31 is the same in every lane
            if (SEG && ((c & ~31) < cb || (c & ~31) >= cend)) continue;
            const bool ok = FULL || (row_ok && c < clim);
            float y[8], src[8];
#pragma unroll
            for (int k = 0; k < 8; k += 2) {                   // z = 0 past the row end (zero-filled copies)
                const float2 yp = __fmul2_rn(f2(inv), make_float2(z[v][k], z[v][k + 1]));
                y[k] = yp.x;
                y[k + 1] = yp.y;
            }
            const uint4 yb = pack8<DT>(y);
            st16_if(a.normed + base + (int64_t)c * 8, yb, normed && ok);
            if (QUANT) {
                if (FROM32) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) src[k] = y[k];
                } else {
                    load8<DT>(yb, src);
                }
                quantize_chunk<FMT, LAYOUT>(src, row, c, ok, FULL || (srow_ok && c < clim), H, a.q, sr, pt.x,
                                            pt.y);
            }
        }
    };
    if (!quant) emit(std::false_type{}, std::false_type{});
    else if (from32) emit(std::true_type{}, std::true_type{});
    else emit(std::true_type{}, std::false_type{});
}

template <int FMT, int LAYOUT, int NV, bool HAS_RES, bool FULL, int DT>
__global__ void __launch_bounds__(kMaxTPR) norm_quant_kernel(const NormArgs a) {
    norm_rows<FMT, LAYOUT, NV, HAS_RES, FULL, DT, !FULL>(a, blockIdx.x);
}

// Shared-memory bytes of the persistent per-token norm: the weight's chunks
// (kept for the CTA's lifetime) and one staging slot a chunk for x.
__host__ __device__ constexpr int norm_pt_persistent_bytes(int nv, int threads) { return nv * 2 * threads * 16; }

// The per-token fused norm of narrow rows at large M (no residual, several
// rows a CTA, exact-fit plans, quantised output) as a persistent grid: one
// wave of CTAs, each taking row blocks blockIdx.x, blockIdx.x + gridDim.x,
// ... The weight is staged once per CTA; a block's x copies go out as soon
// as the previous block's first pass has consumed its slots, so they are in
// flight during that block's reduction, scale and output pass; z stays in
// registers. Every value is formed by the same operations in the same order
// as norm_rows computes it for the per-token format, so the outputs are
// norm_quant_kernel's bit for bit.
template <int NV, int DT>
__global__ void __launch_bounds__(kMaxTPR) norm_pt_persistent_kernel(const NormArgs a) {
    extern __shared__ uint4 stage[];
    __shared__ float2 part[2][32];           // alternate rounds: no barrier needed between blocks
    const int tpr = a.tpr;
    const int nt = blockDim.x;
    const int lrow = threadIdx.x / tpr;
    const int t = threadIdx.x - lrow * tpr;
    const int H = a.H;
    const int64_t nblk = a.M / a.rpc;
    auto wslot = [&](int v) { return &stage[v * nt + threadIdx.x]; };
    auto xslot = [&](int v) { return &stage[(NV + v) * nt + threadIdx.x]; };
    auto issue = [&](int64_t blk) {          // one commit group per chunk
        const int64_t row = blk * a.rpc + lrow;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            cp_async16(xslot(v), a.x + row * a.ldx + (int64_t)(t + v * tpr) * 8, 16);
            cp_async_commit();
        }
    };

    // the weight (not written by the grid this launch may overlap) before pdl_wait
#pragma unroll
    for (int v = 0; v < NV; ++v) cp_async16_cached(wslot(v), a.w + (int64_t)(t + v * tpr) * 8, 16);
    cp_async_commit();
    pdl_wait();
    if ((int64_t)blockIdx.x < nblk) issue(blockIdx.x);
    pdl_trigger();

    const bool from32 = (a.flags & F_FROM_FP32) != 0;
    const float w_add = (a.flags & F_GEMMA) ? 1.0f : -0.0f;
    const bool normed = a.normed != nullptr;
    int round = 0;
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x, round ^= 1) {
        const int64_t row = blk * a.rpc + lrow;
        const int64_t base = row * (int64_t)H;
        float z[NV][8];
        float2 ss2 = make_float2(0.0f, 0.0f);
        float zmax = 0.0f;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            float h[8], wf[8];
            cp_async_wait_group_of<NV>(v);
            load8<DT>(ld_smem16(xslot(v)), h);
            load8<DT>(ld_smem16(wslot(v)), wf);
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                const float2 hp = make_float2(h[k], h[k + 1]);
                const float2 wp = __fadd2_rn(make_float2(wf[k], wf[k + 1]), f2(w_add));
                ss2 = __ffma2_rn(hp, hp, ss2);
                const float2 zp = __fmul2_rn(hp, wp);
                z[v][k] = zp.x;
                z[v][k + 1] = zp.y;
                zmax = fmaxf(zmax, fmaxf(fabsf(zp.x), fabsf(zp.y)));
            }
        }
        // this thread's slots are read: the next block's copies go out now
        if (blk + gridDim.x < nblk) issue(blk + gridDim.x);

        // A one-warp row needs no shared-memory round: row_reduce_sum_max's
        // butterfly over the warp's partials and 31 zeros gives s + 0 and
        // max(m, 0), formed here directly (in this kernel alone: the branch
        // in the shared helper slowed the other kernels).
        float2 r;
        if (tpr == 32) {
            const float sw = warp_sum(ss2.x + ss2.y), mw = warp_max_redux(zmax);
            r = make_float2(sw + 0.0f, fmaxf(mw, 0.0f));
        } else {
            r = row_reduce_sum_max(ss2.x + ss2.y, zmax, part[round], tpr, lrow);
        }
        const float inv = __frsqrt_rn(__fdiv_rn(r.x, (float)H) + a.eps);
        const float ymax = inv * r.y;
        const float2 pt = per_token_scale(from32 ? ymax : round_io<DT>(ymax));
        const ScaleRow sr = scale_row<FMT_PT, SCALE_ROW_MAJOR>(a.so, row);
        auto emit = [&](auto from32_tag) {
            constexpr bool FROM32 = decltype(from32_tag)::value;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int c = t + v * tpr;
                float y[8], src[8];
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    const float2 yp = __fmul2_rn(f2(inv), make_float2(z[v][k], z[v][k + 1]));
                    y[k] = yp.x;
                    y[k + 1] = yp.y;
                }
                const uint4 yb = pack8<DT>(y);
                st16_if(a.normed + base + (int64_t)c * 8, yb, normed);
                if (FROM32) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) src[k] = y[k];
                } else {
                    load8<DT>(yb, src);
                }
                quantize_chunk<FMT_PT, SCALE_ROW_MAJOR>(src, row, c, true, true, H, a.q, sr, pt.x, pt.y);
            }
        };
        if (from32) emit(std::true_type{});
        else emit(std::false_type{});
    }
}

// All-reduce + residual add + RMSNorm + quantisation: x is the sum of
// aa.ar.n partial inputs (AR above); bf16 rows. The bounds-checked kernels
// may split rows into column segments at small M, as the plain norm does
// (each segment's CTA sums the partials of the whole row for the sum of
// squares, and writes its own columns).
template <int FMT, int LAYOUT, int NV, bool HAS_RES, bool FULL>
__global__ void __launch_bounds__(kMaxTPR) norm_ar_kernel(const NormARArgs aa) {
    norm_rows<FMT, LAYOUT, NV, HAS_RES, FULL, DT_BF16, !FULL, false, true>(aa.a, blockIdx.x, &aa.ar);
}

// Bytes of dynamic shared memory the all-reduce norm stages its loads in.
__host__ __device__ constexpr int norm_ar_stage_bytes(bool has_res, int nparts, int nv, int threads) {
    return nv * (norm_stage_inputs(has_res) - 1 + nparts) * threads * 16;
}

// Rows wider than one CTA covers: a cluster of gridDim.x / M CTAs a row
// (cluster dimension set at launch), CTA k of the cluster taking the row's
// k-th column segment; four chunks a thread, bounds always checked.
template <int FMT, int LAYOUT, bool HAS_RES, int DT>
__global__ void __launch_bounds__(kMaxTPR) norm_cluster_kernel(const NormArgs a) {
    norm_rows<FMT, LAYOUT, kMaxNV, HAS_RES, false, DT, false, true>(a, blockIdx.x / cluster_ctas());
}

// Two independent row sets normed in one launch (the q and kv latent norms
// of multi-head latent attention): CTAs [0, grid0) run seg[0], the rest
// seg[1]. Both segments use the CTA size blockDim.x = rpc * tpr of their own
// plan; no residual; bounds always checked.
struct DualArgs {
    NormArgs seg[2];
    int64_t grid0;
};

template <int FMT, int NV, int DT>
__global__ void __launch_bounds__(kMaxTPR) norm_dual_kernel(const DualArgs d) {
    const bool second = blockIdx.x >= d.grid0;
    const NormArgs a = second ? d.seg[1] : d.seg[0];
    norm_rows<FMT, SCALE_ROW_MAJOR, NV, false, false, DT>(a, second ? blockIdx.x - d.grid0 : blockIdx.x);
}

// The activation of one chunk of 8 (gate, up) values, in fp32:
//   OAI:  g' = min(g, limit), u' = min(max(u, -limit), limit),
//         a = (g' * sigmoid(alpha * g')) * (u' + beta). The sigmoid's
//         argument is alpha * clamp(g', glo, ghi), with [glo, ghi] the g'
//         that alpha maps into [kSigLo, kSigHi] (where the clamp acts, the
//         sigmoid of the clamped argument already equals the true one in
//         fp32: 0 or 1); alpha enters the sigmoid's exponent through
//         khi + klo = -alpha log2(e) (two fp32 parts from the host);
//   SiLU: a = (g * sigmoid(g)) * u, the first factor rounded to bf16 when
//         ROUND is set.
// CLAMPED (OAI only): g and u arrive already clamped to limit (g' and u'),
// and alpha > 0 with alpha * limit <= 2^100, so g' bounds the sigmoid's
// argument from above (sigmoid8 is exact there for any argument below
// 2^120) and only the lower clamp remains; the caller has tested the packed
// bf16 gates against the sigmoid's far-negative tail (`rare`), and the
// lower clamp is applied only where that tail is reached. (Clamping g from below on the
// packed bf16 words as well measured 8-17% slower at decode sizes: the
// second dependent bf16x2 min/max lengthens the critical path.)
template <int ACT, bool CLAMPED = false, bool ROUND = false>
__device__ __forceinline__ void activation8(const float (&g)[8], const float (&u)[8], float khi, float klo,
                                            float beta, float limit, float glo, float ghi, float (&a)[8],
                                            bool rare = true) {
    float sg[8];
    if (ACT == ACT_OAI) {
        float gc[8], gs[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            gc[k] = CLAMPED ? g[k] : fminf(g[k], limit);
            gs[k] = CLAMPED ? gc[k] : fmaxf(fminf(gc[k], ghi), glo);
        }
        if (CLAMPED) sigmoid8_prechecked(gs, khi, klo, glo, rare, sg);  // sigmoid(alpha * max(g', glo))
        else sigmoid8(gs, khi, klo, sg);                                 // sigmoid(alpha * gs)
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float2 uc = CLAMPED ? make_float2(u[k], u[k + 1])
                                      : make_float2(fminf(fmaxf(u[k], -limit), limit), fminf(fmaxf(u[k + 1], -limit), limit));
            const float2 r = __fmul2_rn(__fmul2_rn(make_float2(gc[k], gc[k + 1]), make_float2(sg[k], sg[k + 1])),
                                        __fadd2_rn(uc, f2(beta)));
            a[k] = r.x;
            a[k + 1] = r.y;
        }
    } else {
        float zc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) zc[k] = fmaxf(fminf(g[k], kSigHi), kSigLo);
        sigmoid8(zc, -kLog2eHi, -kLog2eLo, sg);
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            float2 s = __fmul2_rn(make_float2(g[k], g[k + 1]), make_float2(sg[k], sg[k + 1]));
            if (ROUND) s = round_bf16x2(s);
            const float2 r = __fmul2_rn(s, make_float2(u[k], u[k + 1]));
            a[k] = r.x;
            a[k + 1] = r.y;
        }
    }
}

// The range of g' that alpha maps into [kSigLo, kSigHi] (everything for alpha = 0).
__device__ __forceinline__ float2 oai_gate_range(float alpha) {
    if (alpha > 0.0f) return make_float2(kSigLo / alpha, kSigHi / alpha);
    if (alpha < 0.0f) return make_float2(kSigHi / alpha, kSigLo / alpha);
    return make_float2(-INFINITY, INFINITY);
}

// One chunk of gate and up from their shared-memory slots, widened to fp32;
// with CLAMP16, g = min(g, limit) and u = clamp(u, -limit, limit) first, on
// the packed bf16 pairs (exact: limit is a bf16 value).
// `rare` (CLAMP16 only): some gate of the chunk lies below a.tail2, where
// the sigmoid's argument reaches its far-negative tail (3 packed min and one
// packed compare for the chunk instead of a test per element).
template <bool CLAMP16>
__device__ __forceinline__ void load_gate_up(const uint4* gs, const uint4* us, const SwigluArgs& a, float (&g)[8],
                                             float (&u)[8], bool& rare) {
    uint4 gw = ld_smem16(gs), uw = ld_smem16(us);
    rare = true;
    if (CLAMP16) {
        gw = make_uint4(bf16x2_min(gw.x, a.lim2), bf16x2_min(gw.y, a.lim2), bf16x2_min(gw.z, a.lim2),
                        bf16x2_min(gw.w, a.lim2));
        uw = make_uint4(bf16x2_max(bf16x2_min(uw.x, a.lim2), a.nlim2), bf16x2_max(bf16x2_min(uw.y, a.lim2), a.nlim2),
                        bf16x2_max(bf16x2_min(uw.z, a.lim2), a.nlim2), bf16x2_max(bf16x2_min(uw.w, a.lim2), a.nlim2));
        rare = bf16x2_any_lt(bf16x2_min(bf16x2_min(gw.x, gw.y), bf16x2_min(gw.z, gw.w)), a.tail2);
    }
    bf16x8_to_f32(gw, g);
    bf16x8_to_f32(uw, u);
}

// Bytes of dynamic shared memory the SwiGLU kernel stages its loads in.
__host__ __device__ constexpr int swiglu_stage_bytes(int nv, int threads) { return nv * 2 * threads * 16; }

// SwiGLU + quantisation. One row per `tpr` threads. Each thread's gate and
// up chunks are copied asynchronously into its own shared-memory slots
// (stage[2v][thread], stage[2v+1][thread]), one commit group per chunk, so
// the whole row is in flight without holding registers and chunk v is
// processed as soon as its own group has landed.
// CLAMP16 (OAI only, see activation8): the limit is a bf16 value and the
// clamps of g and u run on the packed bf16 pairs before widening.
// Column segments: the bounds-checked kernels may run each row as gridDim.y
// CTAs, CTA y taking chunks [y * segc, min((y + 1) * segc, I / 8)), a whole
// number of scale groups (the MX and 1x128 formats have nothing row-wide).
// Chunk indices stay the row's own, so every address and scale index is
// unchanged.
// CL (per-token only): a row wider than one CTA covers, split over the CTAs
// of a cluster, one row per cluster: CTA k takes chunks
// [k * segc, min((k + 1) * segc, I / 8)), and the CTAs' amaxes are combined
// through shared memory (cluster_combine) into the row's scale.
template <int FMT, int LAYOUT, int NV, int ACT, bool FULL, bool CLAMP16, bool CL = false>
__device__ __forceinline__ void swiglu_rows(const SwigluArgs& a) {
    extern __shared__ uint4 stage[];
    __shared__ float part_amax[32];
    const int tpr = a.tpr;
    const int nt = blockDim.x;
    const int lrow = threadIdx.x / tpr;
    const int t = threadIdx.x - lrow * tpr;
    const int64_t row = CL ? (int64_t)(blockIdx.x / cluster_ctas()) : (int64_t)blockIdx.x * a.rpc + lrow;
    const bool row_ok = FULL || row < a.M;
    const int I = a.I, nchunks = I >> 3;
    const uint16_t* grow = a.gu + row * (int64_t)(2 * I);
    const int cb = FULL ? 0 : (int)(CL ? cluster_rank() : blockIdx.y) * a.segc;   // the segment's first chunk
    const int cend = FULL ? nchunks : min(cb + a.segc, nchunks);

    pdl_wait();
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int c = cb + t + v * tpr;
        const bool ok = FULL || (row_ok && c < cend);      // else zero-fill, reading nothing
        cp_async16(&stage[(2 * v) * nt + threadIdx.x], ok ? (const void*)(grow + (int64_t)c * 8) : (const void*)a.gu,
                   ok ? 16 : 0);
        cp_async16(&stage[(2 * v + 1) * nt + threadIdx.x],
                   ok ? (const void*)(grow + I + (int64_t)c * 8) : (const void*)a.gu, ok ? 16 : 0);
        cp_async_commit();
    }
    pdl_trigger();
    if (CL) cluster_arrive_relaxed();       // completed in cluster_combine, once the whole cluster runs

    const bool round_silu = (a.flags & F_ACT_BF16) != 0, from32 = (a.flags & F_FROM_FP32) != 0;
    const float2 gr = oai_gate_range(a.alpha);
    const bool srow_ok = FULL || row < a.so.Ms;
    const ScaleRow sr = scale_row<FMT, LAYOUT>(a.so, row);
    // The chunk loops, specialised by output mode (0: the bf16 activation,
    // no quantisation; 1: quantise the fp32 activation; 2: quantise its bf16
    // rounding) and SiLU's bf16 rounding, so that no per-chunk branch remains.
    auto body = [&](auto mode_tag, auto round_tag) {
        constexpr int MODE = decltype(mode_tag)::value;
        constexpr bool ROUND = decltype(round_tag)::value;
        if (FMT != FMT_PT) {           // MX and 1x128: chunk by chunk, as each lands
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int c = cb + t + v * tpr;
                const bool ok = FULL || (row_ok && c < cend);
                float g[8], u[8], src[8];
                bool rare;
                cp_async_wait_group_of<NV>(v);
                load_gate_up<CLAMP16>(&stage[(2 * v) * nt + threadIdx.x], &stage[(2 * v + 1) * nt + threadIdx.x], a,
                                      g, u, rare);
                activation8<ACT, CLAMP16, ROUND>(g, u, a.khi, a.klo, a.beta, a.limit, gr.x, gr.y, src, rare);
                if (MODE == 0) {
                    st16_if(a.out + row * I + (int64_t)c * 8, f32x8_to_bf16x8(src), ok);
                } else {
                    if (MODE == 2) {
#pragma unroll
                        for (int k = 0; k < 8; k += 2) {
                            const float2 r = round_bf16x2(make_float2(src[k], src[k + 1]));
                            src[k] = r.x;
                            src[k + 1] = r.y;
                        }
                    }
                    // chunks past the row end loaded zeros, and every activation of 0 and 0 is 0
                    quantize_chunk<FMT, LAYOUT>(src, row, c, ok, FULL || (srow_ok && c < cend), I, a.q, sr);
                }
            }
        } else {                       // per-token: the whole row, then its amax
            float src[NV][8];
            float m = 0.0f;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float g[8], u[8];
                bool rare;
                cp_async_wait_group_of<NV>(v);
                load_gate_up<CLAMP16>(&stage[(2 * v) * nt + threadIdx.x], &stage[(2 * v + 1) * nt + threadIdx.x], a,
                                      g, u, rare);
                activation8<ACT, CLAMP16, ROUND>(g, u, a.khi, a.klo, a.beta, a.limit, gr.x, gr.y, src[v], rare);
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    if (MODE == 2) {
                        const float2 r = round_bf16x2(make_float2(src[v][k], src[v][k + 1]));
                        src[v][k] = r.x;
                        src[v][k + 1] = r.y;
                    }
                    m = fmaxf(m, fmaxf(fabsf(src[v][k]), fabsf(src[v][k + 1])));
                }
            }
            if (MODE == 0) {           // (the bf16-out launches use the MX kernels; kept complete here)
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int c = cb + t + v * tpr;
                    st16_if(a.out + row * I + (int64_t)c * 8, f32x8_to_bf16x8(src[v]), FULL || (row_ok && c < cend));
                }
                if (CL) cluster_wait();   // completes the arrive above
                return;
            }
            float amax = row_reduce<true>(m, part_amax, tpr, lrow);
            if (CL) {                  // the row's amax over the cluster
                __shared__ float2 cl_slots[kMaxCluster];
                amax = cluster_combine(make_float2(0.0f, amax), cl_slots).y;
            }
            const float2 pt = per_token_scale(amax);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int c = cb + t + v * tpr;
                quantize_chunk<FMT, LAYOUT>(src[v], row, c, FULL || (row_ok && c < cend),
                                            FULL || (srow_ok && c < cend), I, a.q, sr, pt.x, pt.y);
            }
        }
    };
    auto by_mode = [&](auto round_tag) {
        if (a.out) body(std::integral_constant<int, 0>{}, round_tag);
        else if (from32) body(std::integral_constant<int, 1>{}, round_tag);
        else body(std::integral_constant<int, 2>{}, round_tag);
    };
    if constexpr (ACT == ACT_SILU) {
        if (round_silu) by_mode(std::true_type{});
        else by_mode(std::false_type{});
    } else {
        by_mode(std::false_type{});
    }
}

template <int FMT, int LAYOUT, int NV, int ACT, bool FULL, bool CLAMP16>
__global__ void __launch_bounds__(kMaxTPR) swiglu_quant_kernel(const SwigluArgs a) {
    swiglu_rows<FMT, LAYOUT, NV, ACT, FULL, CLAMP16>(a);
}

// The same with at most 56 registers a thread, which lets three 384-thread
// CTAs share an SM: SiLU-and-mul + 1x128 at I = 12288 measured 11% faster.
// (The OAI kernels measured no better capped inside the prefill step, and
// the per-token kernels keep the whole row in registers.)
template <int FMT, int LAYOUT, int NV, int ACT, bool FULL, bool CLAMP16>
__global__ void __maxnreg__(56) swiglu_quant_kernel_r56(const SwigluArgs a) {
    swiglu_rows<FMT, LAYOUT, NV, ACT, FULL, CLAMP16>(a);
}

// Per-token SwiGLU rows wider than one CTA covers: a cluster of
// gridDim.x / M CTAs a row; four chunks a thread, bounds always checked.
template <int ACT, bool CLAMP16>
__global__ void __launch_bounds__(kMaxTPR) swiglu_pt_cluster_kernel(const SwigluArgs a) {
    swiglu_rows<FMT_PT, SCALE_ROW_MAJOR, kMaxNV, ACT, false, CLAMP16, true>(a);
}

// Bytes of dynamic shared memory the standalone quant kernel stages its loads in.
__host__ __device__ constexpr int quant_stage_bytes(int nv, int threads) { return nv * threads * 16; }

// Standalone FP8 quantisation of 16-bit rows (the quant of the unfused
// chains). Same row engine and quantiser as the fused kernels; the source is
// the bf16 (DT_BF16) or fp16 (DT_F16) value itself. The bounds-checked
// kernels may split rows into gridDim.y column segments (MX and 1x128: CTA y
// takes chunks [y * segc, min((y + 1) * segc, W / 8))); CL (per-token): a row
// wider than one CTA covers, split over the CTAs of a cluster, the amaxes
// combined through shared memory.
template <int FMT, int LAYOUT, int NV, bool FULL, int DT, bool CL = false>
__device__ __forceinline__ void quant_rows(const QuantArgs& a) {
    extern __shared__ uint4 stage[];
    __shared__ float part_amax[32];
    const int tpr = a.tpr;
    const int nt = blockDim.x;
    const int lrow = threadIdx.x / tpr;
    const int t = threadIdx.x - lrow * tpr;
    const int64_t row = CL ? (int64_t)(blockIdx.x / cluster_ctas()) : (int64_t)blockIdx.x * a.rpc + lrow;
    const bool row_ok = FULL || row < a.M;
    const int W = a.W, nchunks = W >> 3;
    const uint16_t* srow = a.src + row * (int64_t)W;
    const int cb = FULL ? 0 : (int)(CL ? cluster_rank() : blockIdx.y) * a.segc;   // the segment's first chunk
    const int cend = FULL ? nchunks : min(cb + a.segc, nchunks);

    pdl_wait();
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int c = cb + t + v * tpr;
        const bool ok = FULL || (row_ok && c < cend);      // else zero-fill, reading nothing
        cp_async16(&stage[v * nt + threadIdx.x], ok ? (const void*)(srow + (int64_t)c * 8) : (const void*)a.src,
                   ok ? 16 : 0);
        cp_async_commit();
    }
    pdl_trigger();
    if (CL) cluster_arrive_relaxed();       // completed in cluster_combine, once the whole cluster runs

    const bool srow_ok = FULL || row < a.so.Ms;
    const ScaleRow sr = scale_row<FMT, LAYOUT>(a.so, row);
    if (FMT != FMT_PT) {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int c = cb + t + v * tpr;
            float src[8];
            cp_async_wait_group_of<NV>(v);
            load8<DT>(ld_smem16(&stage[v * nt + threadIdx.x]), src);
            quantize_chunk<FMT, LAYOUT>(src, row, c, FULL || (row_ok && c < cend), FULL || (srow_ok && c < cend), W,
                                        a.q, sr);
        }
    } else {
        float src[NV][8];
        float m = 0.0f;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            cp_async_wait_group_of<NV>(v);
            load8<DT>(ld_smem16(&stage[v * nt + threadIdx.x]), src[v]);
#pragma unroll
            for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(src[v][k]));
        }
        float amax = row_reduce<true>(m, part_amax, tpr, lrow);
        if (CL) {                              // the row's amax over the cluster
            __shared__ float2 cl_slots[kMaxCluster];
            amax = cluster_combine(make_float2(0.0f, amax), cl_slots).y;
        }
        const float2 pt = per_token_scale(amax);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int c = cb + t + v * tpr;
            quantize_chunk<FMT, LAYOUT>(src[v], row, c, FULL || (row_ok && c < cend), FULL || (srow_ok && c < cend),
                                        W, a.q, sr, pt.x, pt.y);
        }
    }
}

template <int FMT, int LAYOUT, int NV, bool FULL, int DT>
__global__ void __launch_bounds__(kMaxTPR) quant_kernel(const QuantArgs a) {
    quant_rows<FMT, LAYOUT, NV, FULL, DT>(a);
}

// Per-token quantisation of rows wider than one CTA covers: a cluster of
// gridDim.x / M CTAs a row; four chunks a thread, bounds always checked.
template <int DT>
__global__ void __launch_bounds__(kMaxTPR) quant_pt_cluster_kernel(const QuantArgs a) {
    quant_rows<FMT_PT, SCALE_ROW_MAJOR, kMaxNV, false, DT, true>(a);
}

}  // namespace sgq
