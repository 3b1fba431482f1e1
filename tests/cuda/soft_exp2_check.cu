// Checks soft_exp2x2 (the polynomial exp2 of the attention softmax, two lanes at once)
// against CUDA's exp2f on a dense grid of [-125, 8] plus special inputs; prints the
// maximum relative error.
#include <cstdio>
#include <cmath>
#include <vector>
#include "../../relative_bias_hybrid_gb300/csrc/common.cuh"

__global__ void k(const float *x, float *a, float *b, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        // lane pairs (x[i], x[n - 1 - i]): both lanes of the paired instructions are checked
        const float2 y = inkattn::soft_exp2x2(make_float2(x[i], x[n - 1 - i]));
        a[i] = y.x;
        b[i] = exp2f(x[i]);
        if (y.y != inkattn::soft_exp2x2(make_float2(x[n - 1 - i], x[i])).x) a[i] = NAN;
    }
}

int main() {
    const int n = 1 << 22;
    std::vector<float> hx(n);
    for (int i = 0; i < n - 3; ++i) hx[i] = -125.f + 133.f * (float)i / (float)(n - 4);
    hx[n - 3] = 0.f; hx[n - 2] = -0.5f; hx[n - 1] = 0.5f;
    float *x, *a, *b;
    cudaMalloc(&x, n * 4); cudaMalloc(&a, n * 4); cudaMalloc(&b, n * 4);
    cudaMemcpy(x, hx.data(), n * 4, cudaMemcpyHostToDevice);
    k<<<(n + 255) / 256, 256>>>(x, a, b, n);
    if (cudaDeviceSynchronize() != cudaSuccess) { printf("cuda error\n"); return 2; }
    std::vector<float> ha(n), hb(n);
    cudaMemcpy(ha.data(), a, n * 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(hb.data(), b, n * 4, cudaMemcpyDeviceToHost);
    double worst = 0; float at = 0;
    long lane_mismatch = 0;                  // the two lanes disagreed on the same input
    for (int i = 0; i < n; ++i) {
        if (std::isnan(ha[i])) { ++lane_mismatch; continue; }
        const double r = std::fabs((double)ha[i] / (double)hb[i] - 1.0);
        if (r > worst) { worst = r; at = hx[i]; }
    }
    // -inf (a masked logit) must give a negligible value
    float ninf = -INFINITY, hres;
    cudaMemcpy(x, &ninf, 4, cudaMemcpyHostToDevice);
    k<<<1, 1>>>(x, a, b, 1);
    cudaMemcpy(&hres, a, 4, cudaMemcpyDeviceToHost);
    printf("max_rel_err %.6e at %.6f neg_inf %.3e lane_mismatch %ld\n", worst, at, hres, lane_mismatch);
    return 0;
}
