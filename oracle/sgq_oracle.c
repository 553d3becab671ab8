/*
 * sgq_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU oracle of the fused pre-GEMM activation
 * epilogue: residual add + RMSNorm, or SwiGLU, followed by FP8 activation
 * quantisation in three formats. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path never does.
 *
 * Everything is computed in fp64 with scalar loops, one row at a time, in the
 * order the operations are defined. bf16 and E4M3 rounding are written from
 * the format definitions (the E4M3 encoder is a brute-force nearest-code
 * search). It shares no code, header or table with the CUDA library.
 *
 * Sources of the definitions:
 *  - "[ROCm][MiniMax-M3.1] Fuse MXFP8 quant into the add+RMSNorm and SwiGLU"
 *    (vllm PR 65478), "Purpose" and "Test Plan / Correctness": the fused
 *    add+Gemma-RMSNorm writes MXFP8 values, E8M0 scales, the bf16 normed rows
 *    and the updated residual, bit-identical to norm -> standalone quant, i.e.
 *    it quantises the bf16-rounded normed row; the fused SwiGLU computes in
 *    fp32 and quantises without the bf16 rounding; scales are row-major
 *    [M, N/32] E8M0 (review: "Scale layout / scheme contract").
 *  - "[Perf] [AMD] qwen3: Fuse the 1x128 FP8 input quant ..." (sglang PR
 *    48043), "Modifications" and "Accuracy Tests": 1x128 group FP8; the fused
 *    norm quantises the fp32 normed value; the fused SiLU-and-mul rounds silu
 *    to bf16 and the product to bf16, like the unfused SiLU-and-mul.
 *  - "[ROCm] Fuse per-token activation quant into RMSNorm ..." (sglang PR
 *    34502), "Change": per-token FP8 with an [m, 1] scale; fp16 activations
 *    stay fp16 (the norm's input, outputs and quant source are then fp16, as
 *    is the reviewed norm of vllm PR 65478, whose bitwise test covers bf16
 *    and fp16).
 *  - The formulas the pages only name: RMSNorm y = h * (mean(h^2) + eps)^-1/2
 *    * (1 + w) (Gemma) or * w; OAI SwiGLU a = min(g,L) * sigmoid(alpha*min(g,L))
 *    * (clamp(u,-L,L) + beta); SiLU-and-mul a = g*sigmoid(g)*u; E4M3 and E8M0
 *    as in the OCP 8-bit floating point and MX specifications; MX scale
 *    exponent floor(log2(amax)) - 8; FP8 scale amax / 448.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Interface values, kept equal to the public header's by the Python binding
 * tests (the two sides do not include each other). */
enum { ORA_MXFP8 = 0, ORA_BLOCK128 = 1, ORA_PER_TOKEN = 2 };
enum { ORA_SWIGLU_OAI = 0, ORA_SILU_MUL = 1 };
enum { ORA_F_GEMMA = 1u << 0, ORA_F_FROM_FP32 = 1u << 1, ORA_F_ACT_ROUND_BF16 = 1u << 2, ORA_F_FP16 = 1u << 5 };

/* Per-element ambiguity flags written to `amb`. ORA_AMB_TIE marks an
 * element of an FP8 group quantised from fp32 whose argument y/s lies within
 * 2^-22 of an E4M3 midpoint. There the normalisation factor cancels from
 * y/s = 448 * (h_j*w_j) / (h_k*w_k) (k the amax element), a ratio of short
 * bf16 products that often equals a midpoint exactly; only the fp32 rounding
 * of the stored scale then picks a side, so either neighbour is a correct
 * rounding of y * 448 / amax. */
enum { ORA_AMB_SRC = 1, ORA_AMB_CODE = 2, ORA_AMB_TIE = 4 };

/* ------------------------------------------------------------------ bf16 */

/* bf16 is the upper half of an IEEE binary32: 1 sign, 8 exponent, 7 fraction bits. */
double ora_bf16_decode(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Distance between adjacent bf16 values at |v| (the unit in the last place). */
static double bf16_ulp(double a) {
    int e2;
    if (a == 0.0) return ldexp(1.0, -133);
    frexp(a, &e2);              /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;             /* floor(log2(a)) */
    if (e < -126) e = -126;     /* subnormals share the spacing of the smallest binade */
    return ldexp(1.0, e - 7);
}

/* Nearest bf16 to v, ties to even, overflow to infinity. */
uint16_t ora_bf16_round(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a)) return sign | 0x7F80;
    double ulp = bf16_ulp(a);
    double n = nearbyint(a / ulp);   /* a / ulp is exact; default mode rounds half to even */
    double r = n * ulp;              /* exactly a bf16 value (or 2^128 -> inf below) */
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* True when v lies within rel*|v| of a value where its bf16 rounding changes. */
static int near_bf16_boundary(double v, double rel) {
    double a = fabs(v);
    if (a == 0.0) return 0;
    double ulp = bf16_ulp(a);
    double mid = (floor(a / ulp) + 0.5) * ulp;
    double lo_mid = mid - ulp;
    return fabs(a - mid) <= rel * a || fabs(a - lo_mid) <= rel * a;
}

/* ------------------------------------------------------------------ fp16 */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits; exponent
 * field 0 holds the subnormals f * 2^-24; field 31 holds inf and NaN. */
double ora_f16_decode(uint16_t b) {
    int e = (b >> 10) & 0x1F, f = b & 0x3FF;
    double v;
    if (e == 0) v = ldexp((double)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp(1024.0 + (double)f, e - 25);
    return (b & 0x8000) ? -v : v;
}

/* Distance between adjacent fp16 values at |v|. */
static double f16_ulp(double a) {
    int e2;
    if (a == 0.0) return ldexp(1.0, -24);
    frexp(a, &e2);
    int e = e2 - 1;
    if (e < -14) e = -14;       /* subnormals share the spacing of the smallest binade */
    return ldexp(1.0, e - 10);
}

/* Nearest fp16 to v, ties to even; results past the largest finite value
 * (65504, reached by everything below the midpoint 65520) are infinite. */
uint16_t ora_f16_round(double v) {
    if (isnan(v)) return 0x7E00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a)) return sign | 0x7C00;
    double ulp = f16_ulp(a);
    double r = nearbyint(a / ulp) * ulp;     /* exact; half to even */
    if (r >= 65536.0) return sign | 0x7C00;
    if (r < ldexp(1.0, -14)) return sign | (uint16_t)(r / ldexp(1.0, -24));
    int e2;
    frexp(r, &e2);
    int e = e2 - 1;                          /* r in [2^e, 2^(e+1)) */
    uint16_t frac = (uint16_t)(ldexp(r, 10 - e) - 1024.0);
    return sign | (uint16_t)((e + 15) << 10) | frac;
}

static int near_f16_boundary(double v, double rel) {
    double a = fabs(v);
    if (a == 0.0) return 0;
    double ulp = f16_ulp(a);
    double mid = (floor(a / ulp) + 0.5) * ulp;
    double lo_mid = mid - ulp;
    return fabs(a - mid) <= rel * a || fabs(a - lo_mid) <= rel * a;
}

/* The 16-bit activation type: bf16, or fp16 when f16 is set. */
static double io_decode(int f16, uint16_t b) { return f16 ? ora_f16_decode(b) : ora_bf16_decode(b); }
static uint16_t io_round(int f16, double v) { return f16 ? ora_f16_round(v) : ora_bf16_round(v); }
static int near_io_boundary(int f16, double v, double rel) {
    return f16 ? near_f16_boundary(v, rel) : near_bf16_boundary(v, rel);
}

/* ------------------------------------------------------------------ E4M3 */

/* OCP E4M3 (FN): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * S.1111.111 is NaN; largest finite 448; smallest subnormal 2^-9. */
double ora_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double mag;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) mag = (m / 8.0) * ldexp(1.0, -6);
    else mag = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return s ? -mag : mag;
}

/* The 127 finite non-negative E4M3 values, decoded once when the library loads. */
static double e4m3_value[0x7F];

__attribute__((constructor)) static void init_e4m3_values(void) {
    for (int c = 0; c <= 0x7E; ++c) e4m3_value[c] = ora_e4m3_decode((uint8_t)c);
}

/* Round to nearest E4M3 by searching all 127 finite non-negative codes; a tie
 * goes to the code with an even mantissa; magnitudes past 448 take 448 (the
 * nearest finite code), i.e. saturating rounding. The sign is copied. */
uint8_t ora_e4m3_encode(double v) {
    if (isnan(v)) return 0x7F;
    double a = fabs(v);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(e4m3_value[c] - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 0x80 : 0));
}

/* True when t lies within rel*|t| of a point where its E4M3 rounding changes
 * (a midpoint between two adjacent finite codes). Callers pass a window four
 * times the scale window: an element's argument t also carries the rounding
 * of its group's scale. */
static int near_e4m3_boundary(double t, double rel) {
    double a = fabs(t);
    for (int c = 0; c < 0x7E; ++c) {
        double mid = 0.5 * (e4m3_value[c] + e4m3_value[c + 1]);
        if (fabs(a - mid) <= rel * a) return 1;
    }
    return 0;
}

/* ------------------------------------------------------------ scales */

/* MX shared exponent for a block: floor(log2(amax)) minus 8 (the largest
 * exponent of E4M3), clamped to the E8M0 range [-127, 127]; amax = 0 -> -127. */
int ora_mx_scale_exp(double amax) {
    if (amax == 0.0) return -127;
    int e2;
    frexp(amax, &e2);
    int e = (e2 - 1) - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* True when amax lies within rel*amax of a power of two. */
static int near_pow2(double amax, double rel) {
    if (amax == 0.0) return 0;
    int e2;
    double f = frexp(amax, &e2);     /* f in [0.5, 1) */
    double lo = ldexp(0.5, e2), hi = ldexp(1.0, e2);
    (void)f;
    return fabs(amax - lo) <= rel * amax || fabs(hi - amax) <= rel * amax;
}

/* Store the E4M3 argument t and the element's ambiguity flags, if asked. */
static void element_flags(double tj, unsigned char src_amb, double* t, unsigned char* amb, double rel) {
    if (t) *t = tj;
    if (amb)
        *amb = (unsigned char)((src_amb ? (ORA_AMB_SRC | ORA_AMB_CODE) : 0) |
                               (near_e4m3_boundary(tj, 4.0 * rel) ? ORA_AMB_CODE : 0));
}

/* Quantise one group of n source values src[] (fp64) into codes q[] and one
 * scale. `pre[]` are the values before the optional bf16 rounding of the
 * source (equal to src when quantising from fp32), used only for the
 * ambiguity flags. Writes t[] = src / scale (the E4M3 rounding argument). */
static void quant_group(int fmt, int from_fp32, int f16, const double* src, const double* pre,
                        const unsigned char* src_amb, long n, uint8_t* q, void* scale_slot,
                        double* t, unsigned char* amb, unsigned char* gamb, double rel) {
    double amax = 0.0, amax_pre = 0.0;
    for (long j = 0; j < n; ++j) {
        if (fabs(src[j]) > amax) amax = fabs(src[j]);
        if (fabs(pre[j]) > amax_pre) amax_pre = fabs(pre[j]);
    }
    /* Is the group's scale decision robust against small changes of amax? */
    int g_amb = 0;
    if (!from_fp32) {
        /* 16-bit source: amax moves only if an element near the top rounds differently. */
        for (long j = 0; j < n; ++j)
            if (src_amb[j] && fabs(pre[j]) >= amax_pre * (1.0 - ldexp(1.0, f16 ? -10 : -7))) g_amb = 1;
    }
    if (fmt == ORA_MXFP8) {
        if (from_fp32 && near_pow2(amax, rel)) g_amb = 1;
        int e = ora_mx_scale_exp(amax);
        *(uint8_t*)scale_slot = (uint8_t)(e + 127);
        for (long j = 0; j < n; ++j) {
            double tj = src[j] * ldexp(1.0, -e);
            q[j] = ora_e4m3_encode(tj);
            element_flags(tj, src_amb[j], t ? t + j : 0, amb ? amb + j : 0, rel);
        }
    } else {
        /* FP8 with an fp32 scale: s = amax / 448 rounded to fp32 (an fp64
         * quotient of two fp32 values rounded once more to fp32 equals the
         * correctly rounded fp32 quotient). amax is fp32 on any fp32 path, so
         * a source computed in fp32 always leaves the scale's last bits open. */
        if (from_fp32) g_amb = 1;
        float s = (float)(amax / 448.0);
        *(float*)scale_slot = s;
        /* The quotient q_src / s is an fp32 quantity (the pages' kernels form
         * it in fp32): the fp64 quotient rounded once to fp32. For an fp32
         * q_src this is exactly the IEEE fp32 quotient, and an exact tie of
         * q_src / s with an E4M3 midpoint stays a tie. */
        for (long j = 0; j < n; ++j) {
            double tj = (s == 0.0f) ? 0.0 : (double)(float)(src[j] / (double)s);
            q[j] = ora_e4m3_encode(tj);
            element_flags(tj, src_amb[j], t ? t + j : 0, amb ? amb + j : 0, rel);
            if (amb && from_fp32 && near_e4m3_boundary(tj, ldexp(1.0, -22))) amb[j] |= ORA_AMB_TIE;
        }
    }
    if (gamb) *gamb = (unsigned char)g_amb;
}

static long group_size(int fmt, long width) {
    return fmt == ORA_MXFP8 ? 32 : fmt == ORA_BLOCK128 ? 128 : width;
}

static void* scale_at(int fmt, void* scale, long index) {
    return fmt == ORA_MXFP8 ? (void*)((uint8_t*)scale + index) : (void*)((float*)scale + index);
}

/* Quantise one row of `width` values. */
static void quant_row(int fmt, int from_fp32, int f16, const double* pre, long width, long row,
                      uint8_t* q, void* scale, double* t, unsigned char* amb, unsigned char* gamb,
                      double rel, double* src, unsigned char* src_amb) {
    for (long j = 0; j < width; ++j) {
        src[j] = from_fp32 ? pre[j] : io_decode(f16, io_round(f16, pre[j]));
        src_amb[j] = (unsigned char)(from_fp32 ? 0 : near_io_boundary(f16, pre[j], rel));
    }
    long gs = group_size(fmt, width), ng = width / gs;
    for (long g = 0; g < ng; ++g) {
        long off = row * width + g * gs;
        quant_group(fmt, from_fp32, f16, src + g * gs, pre + g * gs, src_amb + g * gs, gs, q + off,
                    scale_at(fmt, scale, row * ng + g), t ? t + off : 0, amb ? amb + off : 0,
                    gamb ? gamb + row * ng + g : 0, rel);
    }
}

/* ------------------------------------------------------- add + RMSNorm */

/*
 * Residual add + RMSNorm + quantisation, one row at a time:
 *   h = x + r                      (r optional; written back rounded to bf16)
 *   y = h / sqrt(sum(h^2)/H + eps) * (1 + w)   (Gemma) or * w (plain)
 *   normed = bf16(y)               (optional output)
 *   quant source = bf16(y), or y itself with ORA_F_FROM_FP32
 * With ORA_F_FP16, x, r, w and the written residual and normed rows are fp16
 * and the rounded quant source is fp16(y).
 * Outputs: q [M,H] E4M3 codes; scale [M,H/32] E8M0 codes, [M,H/128] fp32 or
 * [M,1] fp32. Optional diagnostics: y64 [M,H] (y in fp64), t64 [M,H] (the
 * E4M3 rounding argument), amb [M,H] and gamb [M,groups] flags for decisions
 * within rel of a rounding boundary. Returns 0, or -1 on a bad argument.
 */
int ora_rmsnorm_add_quant(int fmt, unsigned flags, long M, long H, float eps,
                          const uint16_t* x, const uint16_t* r, const uint16_t* w,
                          uint16_t* r_out, uint16_t* normed_out, uint8_t* q, void* scale,
                          double* y64, double* t64, unsigned char* amb, unsigned char* gamb,
                          double rel) {
    if (fmt < 0 || fmt > 2 || M < 0 || H <= 0 || H % group_size(fmt, H) != 0) return -1;
    double* h = (double*)malloc(sizeof(double) * (size_t)H * 3);
    unsigned char* sa = (unsigned char*)malloc((size_t)H);
    if (!h || !sa) { free(h); free(sa); return -1; }
    double *y = h + H, *src = h + 2 * H;
    const int f16 = (flags & ORA_F_FP16) != 0;
    for (long i = 0; i < M; ++i) {
        const uint16_t* xi = x + i * H;
        for (long j = 0; j < H; ++j) h[j] = io_decode(f16, xi[j]) + (r ? io_decode(f16, r[i * H + j]) : 0.0);
        if (r && r_out)
            for (long j = 0; j < H; ++j) r_out[i * H + j] = io_round(f16, h[j]);
        double ss = 0.0;
        for (long j = 0; j < H; ++j) ss += h[j] * h[j];
        double inv = 1.0 / sqrt(ss / (double)H + (double)eps);
        for (long j = 0; j < H; ++j) {
            double wj = io_decode(f16, w[j]);
            y[j] = h[j] * inv * ((flags & ORA_F_GEMMA) ? 1.0 + wj : wj);
        }
        if (normed_out)
            for (long j = 0; j < H; ++j) normed_out[i * H + j] = io_round(f16, y[j]);
        if (y64) memcpy(y64 + i * H, y, sizeof(double) * (size_t)H);
        if (q) quant_row(fmt, (flags & ORA_F_FROM_FP32) != 0, f16, y, H, i, q, scale, t64, amb, gamb, rel, src, sa);
    }
    free(h);
    free(sa);
    return 0;
}

/* ---------------------------------------------------------------- SwiGLU */

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/*
 * SwiGLU + quantisation. gate_up is [M, 2I]: gate = columns [0, I), up =
 * columns [I, 2I) (the two halves of the fused gate/up projection).
 *   OAI:  g' = min(g, limit), u' = min(max(u, -limit), limit),
 *         a = g' * sigmoid(alpha * g') * (u' + beta)
 *   SiLU: a = (g * sigmoid(g)) * u; with ORA_F_ACT_ROUND_BF16 the factor
 *         g*sigmoid(g) is rounded to bf16 before the product.
 * The quant source is bf16(a), or a itself with ORA_F_FROM_FP32.
 * Outputs and diagnostics as for ora_rmsnorm_add_quant (a64 holds a).
 */
int ora_swiglu_quant(int fmt, int act, unsigned flags, long M, long I, float alpha, float beta,
                     float limit, const uint16_t* gate_up, uint8_t* q, void* scale, double* a64,
                     double* t64, unsigned char* amb, unsigned char* gamb, double rel) {
    if (fmt < 0 || fmt > 2 || (act != ORA_SWIGLU_OAI && act != ORA_SILU_MUL) || M < 0 || I <= 0 ||
        I % group_size(fmt, I) != 0)
        return -1;
    double* a = (double*)malloc(sizeof(double) * (size_t)I * 2);
    unsigned char* sa = (unsigned char*)malloc((size_t)I);
    unsigned char* act_amb = (unsigned char*)calloc((size_t)I, 1);
    if (!a || !sa || !act_amb) { free(a); free(sa); free(act_amb); return -1; }
    double* src = a + I;
    for (long i = 0; i < M; ++i) {
        const uint16_t* row = gate_up + i * 2 * I;
        for (long j = 0; j < I; ++j) {
            double g = ora_bf16_decode(row[j]), u = ora_bf16_decode(row[I + j]);
            if (act == ORA_SWIGLU_OAI) {
                double gc = fmin(g, (double)limit);
                double uc = fmin(fmax(u, -(double)limit), (double)limit);
                a[j] = gc * sigmoid((double)alpha * gc) * (uc + (double)beta);
            } else {
                double s = g * sigmoid(g);
                if (flags & ORA_F_ACT_ROUND_BF16) {
                    act_amb[j] = (unsigned char)near_bf16_boundary(s, rel);
                    s = ora_bf16_decode(ora_bf16_round(s));
                }
                a[j] = s * u;
            }
        }
        if (a64) memcpy(a64 + i * I, a, sizeof(double) * (size_t)I);
        quant_row(fmt, (flags & ORA_F_FROM_FP32) != 0, 0, a, I, i, q, scale, t64, amb, gamb, rel, src, sa);
        if (act_amb && (flags & ORA_F_ACT_ROUND_BF16)) {
            /* A rounding of silu(g) that may go either way also leaves the
             * element and (if it is near the top) the group scale open. */
            long gs = group_size(fmt, I), ng = I / gs;
            for (long g = 0; g < ng; ++g) {
                double amax = 0.0;
                for (long j = g * gs; j < (g + 1) * gs; ++j) amax = fmax(amax, fabs(a[j]));
                for (long j = g * gs; j < (g + 1) * gs; ++j) {
                    if (!act_amb[j]) continue;
                    if (amb) amb[i * I + j] |= ORA_AMB_SRC | ORA_AMB_CODE;
                    if (gamb && fabs(a[j]) >= amax * (1.0 - ldexp(1.0, -6))) gamb[i * ng + g] = 1;
                }
            }
        }
    }
    free(a);
    free(sa);
    free(act_amb);
    return 0;
}

/* ------------------------------------------------------- standalone quant */

/*
 * Quantisation of bf16 rows src [M, W] (the standalone quant of the unfused
 * chains: "[ROCm][MiniMax-M3.1] Fuse MXFP8 quant ..." (vllm PR 65478),
 * microbenchmark script (norm, then a separate MXFP8 quant); "[ROCm] Fuse
 * per-token activation quant into RMSNorm ..." (sglang PR 34502),
 * "Motivation" (the standalone per-token quant)). The source values are the
 * bf16 values themselves (fp16 values with ORA_F_FP16). Outputs and
 * diagnostics as above.
 */
int ora_quantize(int fmt, unsigned flags, long M, long W, const uint16_t* src_bits, uint8_t* q, void* scale,
                 double* t64, unsigned char* amb, unsigned char* gamb, double rel) {
    if (fmt < 0 || fmt > 2 || M < 0 || W <= 0 || W % group_size(fmt, W) != 0) return -1;
    double* v = (double*)malloc(sizeof(double) * (size_t)W * 2);
    unsigned char* sa = (unsigned char*)malloc((size_t)W);
    if (!v || !sa) { free(v); free(sa); return -1; }
    for (long i = 0; i < M; ++i) {
        const int f16 = (flags & ORA_F_FP16) != 0;
        for (long j = 0; j < W; ++j) v[j] = io_decode(f16, src_bits[i * W + j]);
        quant_row(fmt, 0, f16, v, W, i, q, scale, t64, amb, gamb, rel, v + W, sa);
    }
    free(v);
    free(sa);
    return 0;
}

/* ------------------------------------------------------------ all-reduce */

/*
 * The all-reduce that precedes the norm under tensor parallelism ("[ROCm]
 * [MiniMax-M3.1] Fuse MXFP8 quant into the add+RMSNorm and SwiGLU"
 * (vllm PR 65478), "Purpose" commit 1: all-reduce + that norm, and
 * "Limitations": a quant-emitting fused all-reduce + norm; "[ROCm] Fuse
 * per-token activation quant into RMSNorm ..." (sglang PR 34502), "Change":
 * the fused all-reduce + RMSNorm + quant of the entry projection). Each of the
 * n ranks holds a partial [count] tensor; the all-reduce's output is their sum
 * in the activation type: out[j] = round(sum_r parts[r][j]), the sum taken in
 * fp64 (exact unless the partials' exponents span more than 45 binades) and
 * rounded once to bf16 (fp16 with ORA_F_FP16). The fused norm then normalises
 * out exactly as ora_rmsnorm_add_quant normalises x. near (optional) flags the
 * elements whose sum lies within rel of a rounding boundary of the activation
 * type, where an fp32 sum may round the other way. Returns 0, or -1 on a bad
 * argument.
 */
int ora_allreduce_sum(int n, const uint16_t* const* parts, long count, unsigned flags, uint16_t* out,
                      unsigned char* near, double rel) {
    if (n < 1 || count < 0 || !parts || !out) return -1;
    const int f16 = (flags & ORA_F_FP16) != 0;
    for (long j = 0; j < count; ++j) {
        double s = 0.0;
        for (int r = 0; r < n; ++r) s += io_decode(f16, parts[r][j]);
        out[j] = io_round(f16, s);
        if (near) near[j] = (unsigned char)near_io_boundary(f16, s, rel);
    }
    return 0;
}
