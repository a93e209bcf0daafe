// Kernels behind qgemm_debug_group_dots: the exact group dots S[m][n][g] are
// read out of the product kernels themselves, one group at a time, by making
// every scale 1 on group g and 0 elsewhere (then y = S[:, :, g] exactly: each
// |S| < 2^19 is a binary32 integer and every other group adds exactly zero).
#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

__global__ void __launch_bounds__(256) fill_ones_kernel(float* __restrict__ v, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        v[i] = 1.0f;
}

// dw[n][j] = binary16(1) if j == g else 0
__global__ void __launch_bounds__(256) one_hot_scales_kernel(uint16_t* __restrict__ dw, int64_t N,
                                                            int64_t G, int64_t g) {
    const int64_t total = N * G;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x)
        dw[i] = (i % G == g) ? (uint16_t)0x3C00u : (uint16_t)0u;
}

// S[m][n][g] = int32(y[m][n]); y holds integers below 2^19 in magnitude
__global__ void __launch_bounds__(256) scatter_group_kernel(const float* __restrict__ y,
                                                           int64_t M, int64_t N, int64_t G,
                                                           int64_t g, int32_t* __restrict__ S) {
    const int64_t total = M * N;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x)
        S[i * G + g] = __float2int_rn(y[i]);
}

int grid_for(int64_t n) {
    int64_t b = (n + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_fill_ones(float* v, int64_t n, cudaStream_t s) {
    fill_ones_kernel<<<grid_for(n), 256, 0, s>>>(v, n);
    return cudaGetLastError();
}

cudaError_t launch_one_hot_scales(uint16_t* dw, int64_t N, int64_t G, int64_t g, cudaStream_t s) {
    one_hot_scales_kernel<<<grid_for(N * G), 256, 0, s>>>(dw, N, G, g);
    return cudaGetLastError();
}

cudaError_t launch_scatter_group(const float* y, int64_t M, int64_t N, int64_t G, int64_t g,
                                 int32_t* S, cudaStream_t s) {
    scatter_group_kernel<<<grid_for(M * N), 256, 0, s>>>(y, M, N, G, g, S);
    return cudaGetLastError();
}

}  // namespace qg
