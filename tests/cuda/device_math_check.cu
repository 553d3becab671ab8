// Test-only kernels around the library's device arithmetic (sigmoid8,
// activation8, div_rn and its packed form div2_rn),
// compiled by tests/test_gpu_device_math.py and compared there against fp64
// and against CUDA's own correctly rounded division.
#include <cuda_runtime.h>

#include "sgq_kernels.cuh"

namespace {

// n must be a multiple of 8.
__global__ void sigmoid_kernel(const float* z, float* out, int n) {
    const int i = 8 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i < n) {
        float zz[8], r[8];
        for (int k = 0; k < 8; ++k) zz[k] = fmaxf(fminf(z[i + k], sgq::kSigHi), sgq::kSigLo);
        sgq::sigmoid8(zz, -sgq::kLog2eHi, -sgq::kLog2eLo, r);
        for (int k = 0; k < 8; ++k) out[i + k] = r[k];
    }
}

// OAI activation through the kernels' own activation8(); n a multiple of 8.
__global__ void oai_kernel(const float* g, const float* u, float* out, int n, float alpha, float beta, float limit) {
    const int i = 8 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i < n) {
        float gg[8], uu[8], r[8];
        for (int k = 0; k < 8; ++k) {
            gg[k] = g[i + k];
            uu[k] = u[i + k];
        }
        const float2 gr = sgq::oai_gate_range(alpha);
        const double kk = -(double)alpha * 1.4426950408889634074;
        const float khi = (float)kk, klo = (float)(kk - (double)khi);
        sgq::activation8<sgq::ACT_OAI>(gg, uu, khi, klo, beta, limit, gr.x, gr.y, r);
        for (int k = 0; k < 8; ++k) out[i + k] = r[k];
    }
}

// The same through the pre-clamped form the packed-bf16 kernels use: g
// clamped to [glo_clamp, limit] and u to limit first (glo_clamp below the
// activation's own lower bound changes nothing), then
// activation8<ACT_OAI, true>.
__global__ void oai_clamped_kernel(const float* g, const float* u, float* out, int n, float alpha, float beta,
                                   float limit, float glo_clamp) {
    const int i = 8 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i < n) {
        float gg[8], uu[8], r[8];
        for (int k = 0; k < 8; ++k) {
            gg[k] = fmaxf(fminf(g[i + k], limit), glo_clamp);
            uu[k] = fminf(fmaxf(u[i + k], -limit), limit);
        }
        const float2 gr = sgq::oai_gate_range(alpha);
        const double kk = -(double)alpha * 1.4426950408889634074;
        const float khi = (float)kk, klo = (float)(kk - (double)khi);
        sgq::activation8<sgq::ACT_OAI, true>(gg, uu, khi, klo, beta, limit, gr.x, gr.y, r);
        for (int k = 0; k < 8; ++k) out[i + k] = r[k];
    }
}

// n must be even: pairs (i, i+1) go through the packed form, each with its
// own divisor, and every element also through the scalar form.
__global__ void div_kernel(const float* a, const float* b, float* q_fast, float* q_pack, float* q_ieee, int n) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i < n) {
        const float r0 = __frcp_rn(b[i]), r1 = __frcp_rn(b[i + 1]);
        q_fast[i] = sgq::div_rn(a[i], b[i], r0);
        q_fast[i + 1] = sgq::div_rn(a[i + 1], b[i + 1], r1);
        const float2 qp = sgq::div2_rn(make_float2(a[i], a[i + 1]), make_float2(-b[i], -b[i + 1]), make_float2(r0, r1));
        q_pack[i] = qp.x;
        q_pack[i + 1] = qp.y;
        q_ieee[i] = __fdiv_rn(a[i], b[i]);
        q_ieee[i + 1] = __fdiv_rn(a[i + 1], b[i + 1]);
    }
}

}  // namespace

extern "C" int run_sigmoid(const float* z, float* out, int n) {
    sigmoid_kernel<<<(n / 8 + 256) / 256, 256>>>(z, out, n);
    return (int)cudaDeviceSynchronize();
}

extern "C" int run_oai(const float* g, const float* u, float* out, int n, float alpha, float beta, float limit) {
    oai_kernel<<<(n / 8 + 256) / 256, 256>>>(g, u, out, n, alpha, beta, limit);
    return (int)cudaDeviceSynchronize();
}

extern "C" int run_oai_clamped(const float* g, const float* u, float* out, int n, float alpha, float beta,
                               float limit, float glo_clamp) {
    oai_clamped_kernel<<<(n / 8 + 256) / 256, 256>>>(g, u, out, n, alpha, beta, limit, glo_clamp);
    return (int)cudaDeviceSynchronize();
}

extern "C" int run_div(const float* a, const float* b, float* q_fast, float* q_pack, float* q_ieee, int n) {
    div_kernel<<<(n / 2 + 255) / 256, 256>>>(a, b, q_fast, q_pack, q_ieee, n);
    return (int)cudaDeviceSynchronize();
}
