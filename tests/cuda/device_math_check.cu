// Test-only kernels around the library's device arithmetic (sigmoid2,
// activation2, div_rn),
// compiled by tests/test_gpu_device_math.py and compared there against fp64
// and against CUDA's own correctly rounded division.
#include <cuda_runtime.h>

#include "sgq_kernels.cuh"

namespace {

__global__ void sigmoid_kernel(const float* z, float* out, int n) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i + 1 < n) {
        const float2 r = sgq::sigmoid2(make_float2(z[i], z[i + 1]), make_float2(0.0f, 0.0f));
        out[i] = r.x;
        out[i + 1] = r.y;
    } else if (i < n) {
        out[i] = sgq::sigmoid2(make_float2(z[i], 0.0f), make_float2(0.0f, 0.0f)).x;
    }
}

// OAI activation of (g, u) pairs through the kernels' own activation2().
__global__ void oai_kernel(const float* g, const float* u, float* out, int n, float alpha, float beta, float limit) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i + 1 < n) {
        const float2 r = sgq::activation2<sgq::ACT_OAI>(make_float2(g[i], g[i + 1]), make_float2(u[i], u[i + 1]),
                                                    alpha, beta, limit, false);
        out[i] = r.x;
        out[i + 1] = r.y;
    }
}

__global__ void div_kernel(const float* a, const float* b, float* q_fast, float* q_ieee, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const float r = __frcp_rn(b[i]);
        q_fast[i] = sgq::div_rn(a[i], b[i], r);
        q_ieee[i] = __fdiv_rn(a[i], b[i]);
    }
}

}  // namespace

extern "C" int run_sigmoid(const float* z, float* out, int n) {
    sigmoid_kernel<<<(n / 2 + 256) / 256, 256>>>(z, out, n);
    return (int)cudaDeviceSynchronize();
}

extern "C" int run_oai(const float* g, const float* u, float* out, int n, float alpha, float beta, float limit) {
    oai_kernel<<<(n / 2 + 256) / 256, 256>>>(g, u, out, n, alpha, beta, limit);
    return (int)cudaDeviceSynchronize();
}

extern "C" int run_div(const float* a, const float* b, float* q_fast, float* q_ieee, int n) {
    div_kernel<<<(n + 255) / 256, 256>>>(a, b, q_fast, q_ieee, n);
    return (int)cudaDeviceSynchronize();
}
