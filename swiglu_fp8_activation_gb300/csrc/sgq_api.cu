// sgq_api.cu -- the C ABI declared in include/sgq.h: host-side argument
// checks, launch planning and one kernel launch per call. Nothing here
// allocates or synchronises; the only state kept between calls is the
// calling thread's last launch error, for sgq_launch_error().
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include <cuda_runtime.h>

#include "sgq.h"
#include "sgq_launch.h"

namespace sgq {

// Rows of width W: `nv` chunks per thread and `tpr` threads per row (a
// multiple of 32, at most kMaxTPR), preferring an exact fit W/8 = tpr * nv.
//  * Large M (bandwidth-bound): the most chunks per thread, so that each
//    thread keeps more loads in flight and rows need fewer threads.
//  * Small M (latency-bound, the whole grid fits in one wave even at one
//    chunk per thread): the fewest chunks per thread, so that each thread's
//    serial work is shortest.
// Several rows share a CTA up to kTargetCTA threads; small M takes fewer rows
// per CTA so that the grid spreads over the SMs.
bool plan_rows(int64_t M, int W, int sm_count, Plan* p) {
    const int nchunks = W / 8;
    const bool small = sm_count > 0 && M * (int64_t)nchunks <= (int64_t)sm_count * 1024;
    int nv = 0, tpr = 0;
    for (int i = 0; i < kMaxNV && nv == 0; ++i) {          // exact fits first
        const int cand = small ? 1 + i : kMaxNV - i;
        if (nchunks % (32 * cand) == 0 && nchunks / cand <= kMaxTPR) {
            nv = cand;
            tpr = nchunks / cand;
        }
    }
    for (int i = 0; i < kMaxNV && nv == 0; ++i) {          // else the fewest threads that cover the row
        const int cand = small ? 1 + i : kMaxNV - i;
        const int t = ((nchunks + cand - 1) / cand + 31) / 32 * 32;
        if (t <= kMaxTPR && (small || (nchunks + 31) / 32 >= cand || cand == 1)) {
            nv = cand;
            tpr = t;
        }
    }
    if (nv == 0 || tpr > kMaxTPR) return false;
    int rpc = kTargetCTA / tpr > 1 ? kTargetCTA / tpr : 1;
    const int64_t per_sm = sm_count > 0 ? (M + sm_count - 1) / sm_count : M;
    if (per_sm < rpc) rpc = per_sm > 1 ? (int)per_sm : 1;
    p->nv = nv;
    p->tpr = tpr;
    p->rpc = rpc;
    p->grid = (M + rpc - 1) / rpc;
    p->full = nchunks == tpr * nv && M % rpc == 0;
    p->sms = sm_count;
    return p->grid <= 0x7FFFFFFF;
}

namespace {
thread_local cudaError_t last_launch_error = cudaSuccess;

// Largest dynamic shared memory granted to each (kernel, device) so far.
std::mutex smem_mu;
std::unordered_map<const void*, int> smem_granted[64];
}  // namespace

void note_launch_error(cudaError_t e) { last_launch_error = e; }

namespace {
struct OccKey {
    const void* k;
    int device, threads, smem;
    bool operator==(const OccKey& o) const {
        return k == o.k && device == o.device && threads == o.threads && smem == o.smem;
    }
};
struct OccHash {
    size_t operator()(const OccKey& o) const {
        return std::hash<const void*>()(o.k) ^ ((size_t)o.device << 48) ^ ((size_t)o.threads << 32) ^ (size_t)o.smem;
    }
};
std::mutex occ_mu;
std::unordered_map<OccKey, int, OccHash> occ_seen;
}  // namespace

cudaError_t ctas_per_sm(const void* kernel, int device, int threads, int smem, int* out) {
    const OccKey key{kernel, device, threads, smem};
    {
        std::lock_guard<std::mutex> lock(occ_mu);
        const auto it = occ_seen.find(key);
        if (it != occ_seen.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    if (smem > 40 * 1024) {
        const cudaError_t e = ensure_dynamic_smem(kernel, device, smem);
        if (e != cudaSuccess) return e;
    }
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, (size_t)smem);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(occ_mu);
    occ_seen[key] = n;
    *out = n;
    return cudaSuccess;
}

cudaError_t ensure_dynamic_smem(const void* kernel, int device, int bytes) {
    if (device < 0 || device >= 64) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    std::lock_guard<std::mutex> lock(smem_mu);
    int& granted = smem_granted[device][kernel];
    if (granted >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) granted = bytes;
    return e;
}

}  // namespace sgq

namespace {

// Largest element count of one tensor: its byte sizes (at most 4 bytes an
// element) stay far inside size_t and the kernels' 64-bit offsets.
constexpr int64_t kMaxElements = int64_t(1) << 56;

bool aligned(const void* p, uintptr_t a) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Half-open byte ranges [a, a+na) and [b, b+nb) intersect (null or empty never does).
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int group_of(int fmt) { return fmt == SGQ_FMT_MXFP8 ? 32 : fmt == SGQ_FMT_FP8_BLOCK128 ? 128 : 8; }

int dt_of(uint32_t flags) { return (flags & SGQ_F_FP16) ? sgq::DT_F16 : sgq::DT_BF16; }

// bf16 bit pattern nearest to a finite float (ties to even), and back.
uint32_t bf16_bits_rn(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

float bf16_value(uint32_t b) {
    const uint32_t u = b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

constexpr uint32_t kLayoutFlags = SGQ_F_SCALE_SWIZZLED | SGQ_F_SCALE_COL_MAJOR;

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// The scale layout the flags select for format fmt at [M, W], and its size
// in bytes. False when a layout flag does not belong to the format.
bool scale_geometry(int fmt, uint32_t flags, int64_t M, int64_t W, sgq::ScaleOut* so, size_t* bytes) {
    const bool swz = (flags & SGQ_F_SCALE_SWIZZLED) != 0, col = (flags & SGQ_F_SCALE_COL_MAJOR) != 0;
    so->ng = (int)(fmt == SGQ_FMT_FP8_PER_TOKEN ? 1 : W / group_of(fmt));
    so->layout = sgq::SCALE_ROW_MAJOR;
    so->ld = so->ng;
    so->Ms = M;
    if (swz && (col || fmt != SGQ_FMT_MXFP8)) return false;
    if (col && fmt != SGQ_FMT_FP8_BLOCK128) return false;
    if (swz) {
        so->layout = sgq::SCALE_SWIZZLED;
        so->ld = round_up(so->ng, 4) / 4;          // 512-byte tiles per 128-row band
        so->Ms = round_up(M, 128);
        *bytes = (size_t)so->Ms * (size_t)round_up(so->ng, 4);
    } else if (col) {
        so->layout = sgq::SCALE_COL_MAJOR;
        so->ld = round_up(M, 4);
        so->Ms = so->ld;
        *bytes = (size_t)so->ng * (size_t)so->ld * 4;
    } else {
        *bytes = (size_t)M * (size_t)so->ng * (fmt == SGQ_FMT_MXFP8 ? 1 : 4);
    }
    return true;
}

// The current device and its multiprocessor count. The count is queried
// once per device and cached; on the call path the one runtime call left is
// cudaGetDevice, which reads the calling thread's current device.
// sgq_set_sm_budget() replaces the count used for planning.
constexpr int kMaxDevices = 64;
std::atomic<int> sm_cache[kMaxDevices];
std::atomic<int> sm_budget{0};

struct Device {
    int id;
    int sms;
};

Device current_device() {
    Device d = {-1, 0};
    if (cudaGetDevice(&d.id) != cudaSuccess) return {-1, 0};
    const int budget = sm_budget.load(std::memory_order_relaxed);
    if (budget > 0) {
        d.sms = budget;
        return d;
    }
    if (d.id < 0 || d.id >= kMaxDevices) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d.id) == cudaSuccess) d.sms = n;
        return d;
    }
    int n = sm_cache[d.id].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d.id) != cudaSuccess) n = 0;
        if (n > 0) sm_cache[d.id].store(n, std::memory_order_relaxed);
    }
    d.sms = n;
    return d;
}

// Plan the rows of a launch whose scale layout covers so.Ms >= M rows: the
// grid covers the layout's padding rows too, and the exact-fit kernels only
// run when there are none.
bool plan_launch(int64_t M, int W, const sgq::ScaleOut& so, const Device& dev, sgq::Plan* p) {
    if (!sgq::plan_rows(so.Ms, W, dev.sms, p)) return false;
    p->full = p->full && so.Ms == M;
    p->device = dev.id;
    return true;
}

// The norms' plan: threads per row and chunks a thread from the real rows M,
// since they fix the order in which a row's sum of squares is added (so a
// scale layout's padding rows change no output value, and the fused norm
// stays equal to rmsnorm_add + quantize_fp8 in every layout); the grid then
// also covers the layout's padding rows [M, Ms).
bool plan_norm(int64_t M, int64_t Ms, int H, int sms, sgq::Plan* p) {
    if (!sgq::plan_rows(M, H, sms, p)) return false;
    if (Ms > M) {
        p->grid = (Ms + p->rpc - 1) / p->rpc;
        p->full = false;
    }
    return p->grid <= 0x7FFFFFFF;
}

// Dynamic shared memory one CTA may use (227 KB on sm_100-class parts).
constexpr int kMaxDynamicSmem = 227 * 1024;

// Chunks (8 columns) one CTA of the row engine covers: kMaxTPR threads with
// kMaxNV chunks each, 16384 columns.
constexpr int kCtaChunks = sgq::kMaxTPR * sgq::kMaxNV;

// A row of nch > kCtaChunks chunks split over a thread block cluster: the
// fewest CTAs that cover it (at most kMaxCluster), each taking segc chunks,
// a multiple of 32 (whole warps, whole scale groups), the last possibly
// fewer; kMaxNV chunks a thread. False when the row needs more CTAs than a
// cluster holds.
bool plan_cluster(int64_t rows, int nch, const Device& dev, sgq::Plan* p, int* segc) {
    int cs = (nch + kCtaChunks - 1) / kCtaChunks;
    if (cs > sgq::kMaxCluster) return false;
    const int sc = (int)round_up((nch + cs - 1) / cs, 32);
    cs = (nch + sc - 1) / sc;
    p->nv = sgq::kMaxNV;
    p->tpr = (int)round_up((sc + sgq::kMaxNV - 1) / sgq::kMaxNV, 32);
    p->rpc = 1;
    p->grid = rows * cs;
    p->full = false;
    p->sms = dev.sms;
    p->seg = 1;
    p->device = dev.id;
    p->cluster = cs;
    *segc = sc;
    return p->grid <= 0x7FFFFFFF;
}

// Column segments (the grid's second dimension) for rows of nch chunks,
// wider than one CTA covers, in a format whose groups are gch chunks and have
// nothing row-wide: the fewest segments that fit a CTA each, at least
// `min_seg`, each a whole number of groups, the last possibly fewer.
int wide_segments(int nch, int gch, int min_seg, int* segc) {
    int s = (nch + kCtaChunks - 1) / kCtaChunks;
    if (s < min_seg) s = min_seg;
    const int sc = (int)round_up((nch + s - 1) / s, gch);
    *segc = sc;
    return (nch + sc - 1) / sc;
}

struct Span {
    const void* p;
    size_t n;
};

// True when any two of the spans intersect.
bool any_overlap(const Span* s, int k) {
    for (int i = 0; i < k; ++i)
        for (int j = i + 1; j < k; ++j)
            if (overlap(s[i].p, s[i].n, s[j].p, s[j].n)) return true;
    return false;
}


int launched(cudaError_t e) {
    if (e == cudaSuccess) return SGQ_OK;
    sgq::note_launch_error(e);
    return SGQ_ERR_LAUNCH;
}

// Column segments a row for a norm launch over `rows` rows (the grid's second
// dimension): while twice the CTAs still fit on the device at one a
// multiprocessor, a row is split in two, up to 8 segments, each a multiple of
// 32 chunks (256 columns; whole warps and whole scale groups) and at least 64
// chunks. Each CTA still reads the whole row of x and r for the sum of
// squares, from L2 at these sizes, but reads the weight and writes the outputs
// of its own segment only: at small M the row's output work and stores then
// spread over several multiprocessors.
int norm_segments(int64_t rows, int64_t H, int sms) {
    if (sms <= 0) return 1;
    const int64_t nch = H / 8;
    int s = 1;
    while (s < 8 && rows * 2 * s <= sms && nch % (64 * s) == 0 && nch / (2 * s) >= 64) s *= 2;
    return s;
}

// The norm launch behind rmsnorm_add_quant (q_out set) and rmsnorm_add
// (q_out null: only the bf16 copy). Width divisibility by the quant group
// and the output pointers required by each entry are checked by the caller.
int norm_call(int fmt, uint32_t flags, int64_t M, int64_t H, float eps, const void* x, const void* residual_in,
              void* residual_out, const void* weight, void* q_out, void* scale_out, void* normed_out,
              sgq_stream_t stream) {
    if (M < 0 || H <= 0 || !(eps >= 0.0f) || isinf(eps)) return SGQ_ERR_INVALID_ARG;
    if (H % 8 != 0 || H > SGQ_MAX_WIDTH) return SGQ_ERR_UNSUPPORTED;
    if (M > kMaxElements / H) return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!x || !weight) return SGQ_ERR_INVALID_ARG;
    if (residual_out && !residual_in) return SGQ_ERR_INVALID_ARG;
    sgq::ScaleOut so;
    size_t sbytes = 0;
    if (!scale_geometry(fmt, flags, M, H, &so, &sbytes)) return SGQ_ERR_INVALID_ARG;
    if (!q_out) sbytes = 0;
    if (!aligned(x, 16) || !aligned(residual_in, 16) || !aligned(residual_out, 16) || !aligned(weight, 16) ||
        !aligned(q_out, 16) || !aligned(normed_out, 16) || !aligned(scale_out, fmt == SGQ_FMT_MXFP8 ? 1 : 4))
        return SGQ_ERR_MISALIGNED;
    const size_t act = (size_t)M * (size_t)H * 2;
    // residual_out == residual_in is the one overlap allowed (in-place update)
    const void* r_out_span = residual_out == residual_in ? nullptr : residual_out;
    const Span spans[] = {{x, act},
                          {residual_in, act},
                          {weight, (size_t)H * 2},
                          {q_out, (size_t)M * H},
                          {scale_out, sbytes},
                          {normed_out, act},
                          {r_out_span, act}};
    if (any_overlap(spans, 7)) return SGQ_ERR_INVALID_ARG;

    // Rows wider than one CTA covers run as a cluster of CTAs a row. Rows too
    // few to fill the device are split into column segments, except for an
    // in-place residual update (another CTA of the row reads r back).
    const Device dev = current_device();
    const int sms = dev.sms;
    sgq::Plan plan;
    int segc = (int)(H / 8);
    const bool wide = H / 8 > kCtaChunks;
    if (wide) {
        if (!plan_cluster(so.Ms, (int)(H / 8), dev, &plan, &segc)) return SGQ_ERR_UNSUPPORTED;
    } else {
        const int seg = residual_out && residual_out == residual_in ? 1 : norm_segments(so.Ms, H, sms);
        if (!plan_norm(M, so.Ms, (int)H, sms, &plan)) return SGQ_ERR_UNSUPPORTED;
        plan.device = dev.id;
        plan.seg = seg;
        plan.full = plan.full && so.Ms == M && seg == 1;   // the exact-fit kernels write whole rows
        segc = (int)(H / 8 / seg);
    }
    sgq::NormArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.r_in = static_cast<const uint16_t*>(residual_in);
    a.r_out = static_cast<uint16_t*>(residual_out);
    a.w = static_cast<const uint16_t*>(weight);
    a.q = static_cast<uint8_t*>(q_out);
    so.p = scale_out;
    a.so = so;
    a.normed = static_cast<uint16_t*>(normed_out);
    a.M = M;
    a.ldx = H;
    a.H = (int)H;
    a.tpr = plan.tpr;
    a.rpc = plan.rpc;
    a.eps = eps;
    a.flags = flags;
    a.segc = segc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Narrow per-token rows at large M (several rows a CTA, at least two waves
    // of row blocks, no residual): the persistent kernel, whose outputs are
    // the row-block kernel's bit for bit (W = 512 at M = 4096: 3.38 -> 2.97 us;
    // W = 1536 at M = 16384: 21.8 -> 18.7 us; with a residual, or at W = 7168,
    // it measured no faster).
    const bool persist = !wide && fmt == SGQ_FMT_FP8_PER_TOKEN && q_out && plan.full && !residual_in &&
                         plan.rpc >= 2 && so.Ms / plan.rpc >= 2 * (int64_t)sms;
    if (persist) return launched(sgq::launch_norm_pt_persistent(dt_of(flags), plan, a, st));
    return launched(wide ? sgq::launch_norm_cluster(fmt, dt_of(flags), plan, a, st)
                         : sgq::launch_norm(fmt, dt_of(flags), plan, a, st));
}

// Column segments a row for a SwiGLU launch over `rows` rows (the grid's
// second dimension), each a whole number of scale groups and at least 512
// columns, at most 16:
//  * few rows: while twice the CTAs still fit on the device at one a
//    multiprocessor, a row is split in two. This spreads a wide row's
//    activation arithmetic (two special-function operations an element)
//    over up to 16 multiprocessors instead of one. (Allowing two CTAs an SM
//    measured slower.)
//  * between half a wave and two waves of rows: the split whose busiest
//    multiprocessor holds the least work (CTAs on it / segments a row), if it
//    beats the whole rows by more than 1/16: SiLU-and-mul at I = 12288 went
//    from 5.04 to 4.03 us at M = 192 (4 segments) and from 5.08 to 4.85 us at
//    M = 256; beyond two waves it measured no better or worse.
// The per-token format needs the row's amax and is never split.
int swiglu_segments(int fmt, int64_t rows, int64_t I, int sms) {
    if (fmt == SGQ_FMT_FP8_PER_TOKEN || sms <= 0) return 1;
    const int64_t nch = I / 8, gch = fmt == SGQ_FMT_FP8_BLOCK128 ? 16 : 4;   // chunks a row, a scale group
    int s = 1;
    while (s < 16 && rows * 2 * s <= sms && nch % (2 * s * gch) == 0 && nch / (2 * s) >= 64) s *= 2;
    if (s == 1 && rows > sms / 2 && rows <= 2 * (int64_t)sms) {
        int64_t best_ctas = (rows + sms - 1) / sms;   // CTAs on the busiest SM, each 1/best_s of a row
        int best_s = 1;
        for (int c = 2; c <= 16; c *= 2) {
            if (nch % (c * gch) != 0 || nch / c < 64) break;
            const int64_t per = (rows * c + sms - 1) / sms;
            if (per * best_s * 16 < best_ctas * c * 15) {
                best_ctas = per;
                best_s = c;
            }
        }
        s = best_s;
    }
    return s;
}

// The SwiGLU launch behind swiglu_quant (q_out set) and swiglu (out set:
// the bf16 activation, no quantisation).
int swiglu_call(int fmt, int act, uint32_t flags, int64_t M, int64_t I, float alpha, float beta, float limit,
                const void* gate_up, void* q_out, void* scale_out, void* out, sgq_stream_t stream) {
    if (act != SGQ_ACT_SWIGLU_OAI && act != SGQ_ACT_SILU_MUL) return SGQ_ERR_INVALID_ARG;
    if ((flags & SGQ_F_ACT_ROUND_BF16) && act != SGQ_ACT_SILU_MUL) return SGQ_ERR_INVALID_ARG;
    if (M < 0 || I <= 0) return SGQ_ERR_INVALID_ARG;
    if (act == SGQ_ACT_SWIGLU_OAI && (!isfinite(alpha) || !isfinite(beta) || !(limit > 0.0f)))
        return SGQ_ERR_INVALID_ARG;
    if (I % 8 != 0 || I > SGQ_MAX_WIDTH) return SGQ_ERR_UNSUPPORTED;
    if (M > kMaxElements / (2 * I)) return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!gate_up) return SGQ_ERR_INVALID_ARG;
    sgq::ScaleOut so;
    size_t sbytes = 0;
    if (!scale_geometry(fmt, flags, M, I, &so, &sbytes)) return SGQ_ERR_INVALID_ARG;
    if (!q_out) sbytes = 0;
    if (!aligned(gate_up, 16) || !aligned(q_out, 16) || !aligned(out, 16) ||
        !aligned(scale_out, fmt == SGQ_FMT_MXFP8 ? 1 : 4))
        return SGQ_ERR_MISALIGNED;
    const Span spans[] = {{gate_up, (size_t)M * I * 4},
                          {q_out, (size_t)M * I},
                          {scale_out, sbytes},
                          {out, (size_t)M * I * 2}};
    if (any_overlap(spans, 4)) return SGQ_ERR_INVALID_ARG;

    // Rows too few to fill the device are split into column segments, and so
    // are rows wider than one CTA covers; per-token rows that wide run as a
    // cluster of CTAs a row (the row's amax is combined across it).
    const Device dev = current_device();
    const int sms = dev.sms;
    const int nch = (int)(I / 8);
    sgq::Plan plan;
    int segc = nch;
    const bool wide = nch > kCtaChunks, cluster = wide && fmt == SGQ_FMT_FP8_PER_TOKEN;
    if (cluster) {
        if (!plan_cluster(so.Ms, nch, dev, &plan, &segc)) return SGQ_ERR_UNSUPPORTED;
    } else {
        int seg = swiglu_segments(fmt, so.Ms, I, sms);
        if (wide) seg = wide_segments(nch, fmt == SGQ_FMT_FP8_BLOCK128 ? 16 : 4, seg, &segc);
        else segc = nch / seg;
        if (!sgq::plan_rows(so.Ms, segc * 8, sms, &plan)) return SGQ_ERR_UNSUPPORTED;
        plan.device = dev.id;
        plan.full = plan.full && so.Ms == M && seg == 1;   // the exact-fit kernels run whole rows
        plan.seg = seg;
    }
    sgq::SwigluArgs a;
    a.gu = static_cast<const uint16_t*>(gate_up);
    a.q = static_cast<uint8_t*>(q_out);
    so.p = scale_out;
    a.so = so;
    a.out = static_cast<uint16_t*>(out);
    a.M = M;
    a.I = (int)I;
    a.segc = segc;
    a.tpr = plan.tpr;
    a.rpc = plan.rpc;
    a.flags = flags;
    a.act = act;
    a.alpha = alpha;
    a.beta = beta;
    a.limit = limit;
    // The OAI clamps run on packed bf16 when the limit is a bf16 value and
    // alpha * limit stays in the range where the sigmoid needs no upper clamp.
    const uint32_t lb = bf16_bits_rn(limit);
    const bool clamp16 = act == SGQ_ACT_SWIGLU_OAI && alpha > 0.0f && isfinite(limit) &&
                         alpha * limit <= 0x1p100f && bf16_value(lb) == limit;
    // -alpha log2(e) in two fp32 parts (head rounded, then the rest)
    const double k = -(double)alpha * 1.4426950408889634074;
    a.khi = (float)k;
    a.klo = (float)(k - (double)a.khi);
    a.lim2 = lb | (lb << 16);
    a.nlim2 = a.lim2 ^ 0x80008000u;
    a.tail2 = 0;
    if (clamp16) {
        // the least bf16 gate t with RN(khi t) <= 125, from the largest bf16
        // not above 125 / khi (khi < 0) upwards: every gate >= t keeps the
        // sigmoid's main formula in range, and only chunks holding a gate
        // below t take the kernel's far-negative branch
        uint32_t tb = bf16_bits_rn((float)(125.0 / (double)a.khi));
        while (bf16_value(tb) * a.khi > 125.0f) tb = (tb & 0x8000u) ? tb - 1 : tb + 1;   // towards +inf
        a.tail2 = tb | (tb << 16);
    }
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return launched(cluster ? sgq::launch_swiglu_pt_cluster(plan, a, clamp16, st)
                            : sgq::launch_swiglu(fmt, plan, a, clamp16, st));
}

int gcd(int a, int b) { return b == 0 ? a : gcd(b, a % b); }

// Plan of the two-segment norm. Each segment keeps the threads per row of
// its own single-norm plan (plan_rows for M and its width), and the launch
// takes the larger of the two plans' chunks a thread (NV): the extra chunks of
// the other segment lie past its row end and add exact zeros, so every thread
// sums the same chunks in the same order as a rmsnorm_add_quant call on that
// segment, and each segment's outputs equal that call's bit for bit. The CTA
// size T is the least common multiple of the two threads per row (so every
// CTA holds whole rows of its segment), grown towards kTargetCTA at large M.
// Where that multiple exceeds kMaxTPR, both segments take the wider one's
// threads per row, and the outputs then match a single call within the
// tolerances only (its sum of squares is added in another order).
bool plan_dual(int64_t M, int Ha, int Hb, int sms, sgq::Plan* p, int tpr[2], int rpc[2], int64_t* grid0) {
    sgq::Plan single[2];
    if (!sgq::plan_rows(M, Ha, sms, &single[0]) || !sgq::plan_rows(M, Hb, sms, &single[1])) return false;
    const int nv = single[0].nv > single[1].nv ? single[0].nv : single[1].nv;
    int t[2] = {single[0].tpr, single[1].tpr};
    int T = t[0] / gcd(t[0], t[1]) * t[1];
    if (T > sgq::kMaxTPR) {
        const int n[2] = {Ha / 8, Hb / 8};
        for (int s = 0; s < 2; ++s) t[s] = ((n[s] + nv - 1) / nv + 31) / 32 * 32;
        T = t[0] > t[1] ? t[0] : t[1];
        if (T > sgq::kMaxTPR) return false;
        t[0] = t[1] = T;
    }
    const bool small = sms > 0 && M * (int64_t)(Ha / 8 + Hb / 8) <= (int64_t)sms * 1024;
    if (!small && T < sgq::kTargetCTA) T *= sgq::kTargetCTA / T;
    for (int s = 0; s < 2; ++s) {
        tpr[s] = t[s];
        rpc[s] = T / t[s];
    }
    *grid0 = (M + rpc[0] - 1) / rpc[0];
    p->nv = nv;
    p->tpr = T;
    p->rpc = 1;
    p->grid = *grid0 + (M + rpc[1] - 1) / rpc[1];
    p->full = false;
    p->sms = sms;
    return p->grid <= 0x7FFFFFFF;
}

}  // namespace

extern "C" {

int sgq_abi_version(void) { return SGQ_ABI_VERSION; }

int sgq_set_sm_budget(int sms) {
    if (sms < 0) return SGQ_ERR_INVALID_ARG;
    sm_budget.store(sms, std::memory_order_relaxed);
    return SGQ_OK;
}

const char* sgq_launch_error(void) {
    return sgq::last_launch_error == cudaSuccess ? "no launch error" : cudaGetErrorString(sgq::last_launch_error);
}

const char* sgq_status_string(int status) {
    switch (status) {
        case SGQ_OK: return "ok";
        case SGQ_ERR_INVALID_ARG: return "invalid argument";
        case SGQ_ERR_UNSUPPORTED: return "unsupported width";
        case SGQ_ERR_MISALIGNED: return "misaligned pointer";
        case SGQ_ERR_LAUNCH: return "kernel launch failed";
        default: return "unknown status";
    }
}

int rmsnorm_add_quant(int fmt, uint32_t flags, int64_t M, int64_t H, float eps, const void* x,
                      const void* residual_in, void* residual_out, const void* weight, void* q_out,
                      void* scale_out, void* normed_out, sgq_stream_t stream) {
    if (fmt < SGQ_FMT_MXFP8 || fmt > SGQ_FMT_FP8_PER_TOKEN) return SGQ_ERR_INVALID_ARG;
    if (flags & ~(SGQ_F_GEMMA_WEIGHT | SGQ_F_QUANT_FROM_FP32 | SGQ_F_FP16 | kLayoutFlags)) return SGQ_ERR_INVALID_ARG;
    if (H > 0 && H % group_of(fmt) != 0) return SGQ_ERR_UNSUPPORTED;
    if (M > 0 && (!q_out || !scale_out)) return SGQ_ERR_INVALID_ARG;
    return norm_call(fmt, flags, M, H, eps, x, residual_in, residual_out, weight, q_out, scale_out, normed_out,
                     stream);
}

int rmsnorm_add(uint32_t flags, int64_t M, int64_t H, float eps, const void* x, const void* residual_in,
                void* residual_out, const void* weight, void* normed_out, sgq_stream_t stream) {
    if (flags & ~(SGQ_F_GEMMA_WEIGHT | SGQ_F_FP16)) return SGQ_ERR_INVALID_ARG;
    if (H > 0 && H % 8 != 0) return SGQ_ERR_UNSUPPORTED;
    if (M > 0 && !normed_out) return SGQ_ERR_INVALID_ARG;
    return norm_call(SGQ_FMT_MXFP8, flags, M, H, eps, x, residual_in, residual_out, weight, nullptr, nullptr,
                     normed_out, stream);
}

int allreduce_rmsnorm_add_quant(int fmt, uint32_t flags, int nranks, int64_t M, int64_t H, float eps,
                                const void* const* partials, const void* residual_in, void* residual_out,
                                const void* weight, void* q_out, void* scale_out, void* normed_out,
                                sgq_stream_t stream) {
    if (fmt < SGQ_FMT_MXFP8 || fmt > SGQ_FMT_FP8_PER_TOKEN) return SGQ_ERR_INVALID_ARG;
    if (flags & ~(SGQ_F_GEMMA_WEIGHT | SGQ_F_QUANT_FROM_FP32 | kLayoutFlags)) return SGQ_ERR_INVALID_ARG;
    if (nranks < 1 || nranks > SGQ_MAX_RANKS || !partials) return SGQ_ERR_INVALID_ARG;
    if (M < 0 || H <= 0 || !(eps >= 0.0f) || isinf(eps)) return SGQ_ERR_INVALID_ARG;
    if (H % group_of(fmt) != 0 || H % 8 != 0 || H / 8 > kCtaChunks) return SGQ_ERR_UNSUPPORTED;
    if (M > kMaxElements / H) return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!weight || !q_out || !scale_out) return SGQ_ERR_INVALID_ARG;
    if (residual_out && !residual_in) return SGQ_ERR_INVALID_ARG;
    for (int r = 0; r < nranks; ++r)
        if (!partials[r]) return SGQ_ERR_INVALID_ARG;
    sgq::ScaleOut so;
    size_t sbytes = 0;
    if (!scale_geometry(fmt, flags, M, H, &so, &sbytes)) return SGQ_ERR_INVALID_ARG;
    for (int r = 0; r < nranks; ++r)
        if (!aligned(partials[r], 16)) return SGQ_ERR_MISALIGNED;
    if (!aligned(residual_in, 16) || !aligned(residual_out, 16) || !aligned(weight, 16) || !aligned(q_out, 16) ||
        !aligned(normed_out, 16) || !aligned(scale_out, fmt == SGQ_FMT_MXFP8 ? 1 : 4))
        return SGQ_ERR_MISALIGNED;
    const size_t act = (size_t)M * (size_t)H * 2;
    const void* r_out_span = residual_out == residual_in ? nullptr : residual_out;
    // outputs may overlap nothing; the inputs (partials, residual, weight) may overlap each other
    const Span outs[] = {{q_out, (size_t)M * H}, {scale_out, sbytes}, {normed_out, act}, {r_out_span, act}};
    if (any_overlap(outs, 4)) return SGQ_ERR_INVALID_ARG;
    for (const Span& o : outs) {
        for (int r = 0; r < nranks; ++r)
            if (overlap(o.p, o.n, partials[r], act)) return SGQ_ERR_INVALID_ARG;
        if (overlap(o.p, o.n, weight, (size_t)H * 2)) return SGQ_ERR_INVALID_ARG;
        if (o.p != r_out_span && overlap(o.p, o.n, residual_in, act)) return SGQ_ERR_INVALID_ARG;
    }
    if (overlap(r_out_span, act, residual_in, act)) return SGQ_ERR_INVALID_ARG;

    // the plain norm's plan and column segments (so the sum of squares is
    // added in the same order as rmsnorm_add_quant's), each partial staged
    const Device dev = current_device();
    // Column segments only at the smallest M: each segment's CTA reads every
    // rank's partial of the whole row, so the reads grow with ranks x
    // segments (TP4 at M = 1 / 8: 2.55 / 2.51 -> 2.13 / 2.20 us with them;
    // TP8 at M = 64: 2.98 -> 3.17 us, slower).
    const int seg = (residual_out && residual_out == residual_in) || so.Ms * nranks > 64
                        ? 1 : norm_segments(so.Ms, H, dev.sms);
    sgq::Plan plan;
    if (!plan_norm(M, so.Ms, (int)H, dev.sms, &plan)) return SGQ_ERR_UNSUPPORTED;
    plan.device = dev.id;
    plan.full = plan.full && so.Ms == M && seg == 1;
    plan.seg = seg;
    if (sgq::norm_ar_stage_bytes(residual_in != nullptr, nranks, plan.nv, plan.rpc * plan.tpr) > kMaxDynamicSmem)
        return SGQ_ERR_UNSUPPORTED;
    sgq::NormARArgs aa;
    sgq::NormArgs& a = aa.a;
    a.x = nullptr;
    a.r_in = static_cast<const uint16_t*>(residual_in);
    a.r_out = static_cast<uint16_t*>(residual_out);
    a.w = static_cast<const uint16_t*>(weight);
    a.q = static_cast<uint8_t*>(q_out);
    so.p = scale_out;
    a.so = so;
    a.normed = static_cast<uint16_t*>(normed_out);
    a.M = M;
    a.ldx = H;
    a.H = (int)H;
    a.tpr = plan.tpr;
    a.rpc = plan.rpc;
    a.eps = eps;
    a.flags = flags;
    a.segc = (int)(H / 8 / seg);
    aa.ar.n = nranks;
    for (int r = 0; r < sgq::kMaxRanks; ++r)
        aa.ar.p[r] = static_cast<const uint16_t*>(partials[r < nranks ? r : 0]);
    return launched(sgq::launch_norm_ar(fmt, plan, aa, static_cast<cudaStream_t>(stream)));
}

int swiglu_quant(int fmt, int act, uint32_t flags, int64_t M, int64_t I, float alpha, float beta,
                 float limit, const void* gate_up, void* q_out, void* scale_out, sgq_stream_t stream) {
    if (fmt < SGQ_FMT_MXFP8 || fmt > SGQ_FMT_FP8_PER_TOKEN) return SGQ_ERR_INVALID_ARG;
    if (flags & ~(SGQ_F_QUANT_FROM_FP32 | SGQ_F_ACT_ROUND_BF16 | kLayoutFlags)) return SGQ_ERR_INVALID_ARG;
    if (I > 0 && I % group_of(fmt) != 0) return SGQ_ERR_UNSUPPORTED;
    if (M > 0 && (!q_out || !scale_out)) return SGQ_ERR_INVALID_ARG;
    return swiglu_call(fmt, act, flags, M, I, alpha, beta, limit, gate_up, q_out, scale_out, nullptr, stream);
}

int swiglu(int act, uint32_t flags, int64_t M, int64_t I, float alpha, float beta, float limit,
           const void* gate_up, void* out, sgq_stream_t stream) {
    if (flags & ~SGQ_F_ACT_ROUND_BF16) return SGQ_ERR_INVALID_ARG;
    if (I > 0 && I % 8 != 0) return SGQ_ERR_UNSUPPORTED;
    if (M > 0 && !out) return SGQ_ERR_INVALID_ARG;
    return swiglu_call(SGQ_FMT_MXFP8, act, flags, M, I, alpha, beta, limit, gate_up, nullptr, nullptr, out, stream);
}

int quantize_fp8(int fmt, uint32_t flags, int64_t M, int64_t W, const void* src, void* q_out, void* scale_out,
                 sgq_stream_t stream) {
    if (fmt < SGQ_FMT_MXFP8 || fmt > SGQ_FMT_FP8_PER_TOKEN) return SGQ_ERR_INVALID_ARG;
    if (flags & ~(kLayoutFlags | SGQ_F_FP16)) return SGQ_ERR_INVALID_ARG;
    if (M < 0 || W <= 0) return SGQ_ERR_INVALID_ARG;
    if (W % group_of(fmt) != 0 || W > SGQ_MAX_WIDTH) return SGQ_ERR_UNSUPPORTED;
    if (M > kMaxElements / W) return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!src || !q_out || !scale_out) return SGQ_ERR_INVALID_ARG;
    sgq::ScaleOut so;
    size_t sbytes = 0;
    if (!scale_geometry(fmt, flags, M, W, &so, &sbytes)) return SGQ_ERR_INVALID_ARG;
    if (!aligned(src, 16) || !aligned(q_out, 16) || !aligned(scale_out, fmt == SGQ_FMT_MXFP8 ? 1 : 4))
        return SGQ_ERR_MISALIGNED;
    const Span spans[] = {{src, (size_t)M * W * 2}, {q_out, (size_t)M * W}, {scale_out, sbytes}};
    if (any_overlap(spans, 3)) return SGQ_ERR_INVALID_ARG;

    // Rows wider than one CTA covers: column segments (MX, 1x128), or a
    // cluster of CTAs a row (per-token, whose scale needs the row's amax).
    const Device dev = current_device();
    const int nch = (int)(W / 8);
    sgq::Plan plan;
    int segc = nch;
    const bool wide = nch > kCtaChunks, cluster = wide && fmt == SGQ_FMT_FP8_PER_TOKEN;
    if (cluster) {
        if (!plan_cluster(so.Ms, nch, dev, &plan, &segc)) return SGQ_ERR_UNSUPPORTED;
    } else if (wide) {
        const int seg = wide_segments(nch, fmt == SGQ_FMT_FP8_BLOCK128 ? 16 : 4, 1, &segc);
        if (!sgq::plan_rows(so.Ms, segc * 8, dev.sms, &plan)) return SGQ_ERR_UNSUPPORTED;
        plan.device = dev.id;
        plan.full = false;
        plan.seg = seg;
    } else {
        if (!plan_launch(M, (int)W, so, dev, &plan)) return SGQ_ERR_UNSUPPORTED;
    }
    sgq::QuantArgs a;
    a.src = static_cast<const uint16_t*>(src);
    a.q = static_cast<uint8_t*>(q_out);
    so.p = scale_out;
    a.so = so;
    a.M = M;
    a.W = (int)W;
    a.tpr = plan.tpr;
    a.rpc = plan.rpc;
    a.segc = segc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return launched(cluster ? sgq::launch_quant_pt_cluster(dt_of(flags), plan, a, st)
                            : sgq::launch_quant(fmt, dt_of(flags), plan, a, st));
}

int rmsnorm_dual_quant(int fmt, uint32_t flags, int64_t M, float eps, const sgq_norm_seg_t* seg_a,
                       const sgq_norm_seg_t* seg_b, sgq_stream_t stream) {
    if (fmt < SGQ_FMT_MXFP8 || fmt > SGQ_FMT_FP8_PER_TOKEN) return SGQ_ERR_INVALID_ARG;
    if (flags & ~(SGQ_F_GEMMA_WEIGHT | SGQ_F_QUANT_FROM_FP32 | SGQ_F_FP16)) return SGQ_ERR_INVALID_ARG;
    if (!seg_a || !seg_b || M < 0 || !(eps >= 0.0f) || isinf(eps)) return SGQ_ERR_INVALID_ARG;
    const sgq_norm_seg_t* sg[2] = {seg_a, seg_b};
    for (int i = 0; i < 2; ++i) {
        const sgq_norm_seg_t& s = *sg[i];
        if (s.H <= 0 || s.ld < s.H) return SGQ_ERR_INVALID_ARG;
        if (s.H % (s.q_out ? group_of(fmt) : 8) != 0 || s.H > SGQ_MAX_DUAL_WIDTH) return SGQ_ERR_UNSUPPORTED;
        if (M > kMaxElements / s.ld) return SGQ_ERR_INVALID_ARG;
    }
    if (M == 0) return SGQ_OK;
    Span in[4], out[6];
    for (int i = 0; i < 2; ++i) {
        const sgq_norm_seg_t& s = *sg[i];
        if (!s.x || !s.weight || (!s.q_out) != (!s.scale_out) || (!s.q_out && !s.normed_out))
            return SGQ_ERR_INVALID_ARG;
        if (s.ld % 8 != 0 || !aligned(s.x, 16) || !aligned(s.weight, 16) || !aligned(s.q_out, 16) ||
            !aligned(s.normed_out, 16) || !aligned(s.scale_out, fmt == SGQ_FMT_MXFP8 ? 1 : 4))
            return SGQ_ERR_MISALIGNED;
        sgq::ScaleOut so;
        size_t sbytes = 0;
        scale_geometry(fmt, 0, M, s.H, &so, &sbytes);
        in[2 * i] = {s.x, (size_t)((M - 1) * s.ld + s.H) * 2};
        in[2 * i + 1] = {s.weight, (size_t)s.H * 2};
        out[3 * i] = {s.q_out, (size_t)(M * s.H)};
        out[3 * i + 1] = {s.scale_out, s.q_out ? sbytes : 0};
        out[3 * i + 2] = {s.normed_out, (size_t)(M * s.H) * 2};
    }
    // outputs may overlap neither each other nor any input; the inputs may
    // overlap (q and kv are often column ranges of one projection output)
    if (any_overlap(out, 6)) return SGQ_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        for (int j = 0; j < 4; ++j)
            if (overlap(out[i].p, out[i].n, in[j].p, in[j].n)) return SGQ_ERR_INVALID_ARG;

    sgq::Plan plan;
    int tpr[2], rpc[2];
    int64_t grid0 = 0;
    const Device dev = current_device();
    if (!plan_dual(M, (int)seg_a->H, (int)seg_b->H, dev.sms, &plan, tpr, rpc, &grid0)) return SGQ_ERR_UNSUPPORTED;
    plan.device = dev.id;
    sgq::DualArgs d;
    for (int i = 0; i < 2; ++i) {
        const sgq_norm_seg_t& s = *sg[i];
        sgq::NormArgs& a = d.seg[i];
        a.x = static_cast<const uint16_t*>(s.x);
        a.r_in = nullptr;
        a.r_out = nullptr;
        a.w = static_cast<const uint16_t*>(s.weight);
        a.q = static_cast<uint8_t*>(s.q_out);
        size_t sbytes = 0;
        scale_geometry(fmt, 0, M, s.H, &a.so, &sbytes);
        a.so.p = s.scale_out;
        a.normed = static_cast<uint16_t*>(s.normed_out);
        a.M = M;
        a.ldx = s.ld;
        a.H = (int)s.H;
        a.tpr = tpr[i];
        a.rpc = rpc[i];
        a.eps = eps;
        a.flags = flags;
        a.segc = (int)(s.H / 8);   // whole rows
    }
    d.grid0 = grid0;
    return launched(sgq::launch_norm_dual(fmt, dt_of(flags), plan, d, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
