// Decode GEMV (M <= 8): y[m,n] = sum_g dw[n,g] dx[m,g] S[m,n,g] for Q8_0 or
// Q4_0 weights, bound by the weight stream from HBM.
//
// The thin-M product is a structural bandwidth problem ("A 35B
// Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU", Results:
// thin-M GEMM is the limit; Methodology 1: a W4A8 integer decode kernel), so
// the kernel is organised around the weight bytes:
//   * a warp streams one weight row (or a K-slice of it) with 16-byte
//     ld.global.nc loads, 512 contiguous bytes per warp per step, several
//     steps in flight per lane;
//   * group dot products are exact int32 sums of dp4a (Q8: a lane holds half a
//     group and the two halves meet through one shuffle; Q4: a lane holds a
//     whole 16-byte group);
//   * each exact S is scaled by dw * dx and added to a binary32 partial;
//   * split-K: the 8 warps of a block cover R rows x W K-slices (R * W = 8);
//     the W binary32 partials of a row meet in shared memory and are summed in
//     slice order, so the result is deterministic for a given shape.  Partial
//     accumulators stay in binary32 (the mining-card page's split-K
//     FlashAttention section: half-precision partials drifted, binary32 ones
//     did not).
#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 4;

template <int M, bool kQ4, int W>
__global__ void __launch_bounds__(256)
gemv_kernel(const int8_t* __restrict__ qx, const float* __restrict__ dx,
            const uint8_t* __restrict__ qw, const uint16_t* __restrict__ dw,
            float* __restrict__ y, int64_t N, int64_t K, int64_t ldy) {
    constexpr int R = kWarps / W;
    __shared__ float part[kWarps][M];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = K / kGroup;
    const int64_t n = (int64_t)blockIdx.x * R + warp / W;
    const int split = warp % W;
    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.f;

    if (n < N) {
        // K-slice of this warp, in whole groups.
        const int64_t gps = (G + W - 1) / W;
        const int64_t g0 = split * gps;
        const int64_t g1 = min(G, g0 + gps);
        const float* dxr = dx;
        const uint16_t* dwr = dw + n * G;
        if (!kQ4) {
            // a lane holds 16 bytes = half a group; a step covers 16 groups
            const uint8_t* wrow = qw + n * K;
            const int64_t b0 = g0 * kGroup, b1 = g1 * kGroup;
            for (int64_t base = b0; base < b1; base += 512 * kUnroll) {
                uint4 wv[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t off = base + u * 512 + lane * 16;
                    wv[u] = off < b1 ? ldg_nc_v4(wrow + off) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t off = base + u * 512 + lane * 16;
                    const bool ok = off < b1;          // same for both lanes of a group
                    const int64_t g = off / kGroup;
                    const float dwf = ok ? half_bits_to_float(dwr[g]) : 0.f;
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        int s = 0;
                        if (ok) {
                            const uint4 xv = ldg_v4(qx + m * K + off);
                            s = dp4a_ss(wv[u].x, xv.x, s);
                            s = dp4a_ss(wv[u].y, xv.y, s);
                            s = dp4a_ss(wv[u].z, xv.z, s);
                            s = dp4a_ss(wv[u].w, xv.w, s);
                        }
                        s += __shfl_xor_sync(0xffffffffu, s, 1);   // exact group sum
                        if (ok && (lane & 1) == 0)
                            acc[m] = fmaf((float)s, dwf * dxr[m * G + g], acc[m]);
                    }
                }
            }
        } else {
            // a lane holds one whole 16-byte group; a step covers 32 groups
            const uint8_t* wrow = qw + n * (K / 2);
            for (int64_t gb = g0; gb < g1; gb += 32 * kUnroll) {
                uint4 wv[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t g = gb + u * 32 + lane;
                    wv[u] = g < g1 ? ldg_nc_v4(wrow + g * 16) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t g = gb + u * 32 + lane;
                    if (g < g1) {
                        const float dwf = half_bits_to_float(dwr[g]);
                        const uint32_t wl[4] = {wv[u].x & 0x0f0f0f0fu, wv[u].y & 0x0f0f0f0fu,
                                                wv[u].z & 0x0f0f0f0fu, wv[u].w & 0x0f0f0f0fu};
                        const uint32_t wh[4] = {(wv[u].x >> 4) & 0x0f0f0f0fu,
                                                (wv[u].y >> 4) & 0x0f0f0f0fu,
                                                (wv[u].z >> 4) & 0x0f0f0f0fu,
                                                (wv[u].w >> 4) & 0x0f0f0f0fu};
#pragma unroll
                        for (int m = 0; m < M; ++m) {
                            const uint4 xa = ldg_v4(qx + m * K + g * kGroup);
                            const uint4 xb = ldg_v4(qx + m * K + g * kGroup + 16);
                            // sum (q+8)*x - 8*sum x, exact in int32
                            int s = dp4a_us(wl[0], xa.x, 0);
                            s = dp4a_us(wl[1], xa.y, s);
                            s = dp4a_us(wl[2], xa.z, s);
                            s = dp4a_us(wl[3], xa.w, s);
                            s = dp4a_us(wh[0], xb.x, s);
                            s = dp4a_us(wh[1], xb.y, s);
                            s = dp4a_us(wh[2], xb.z, s);
                            s = dp4a_us(wh[3], xb.w, s);
                            int sx = dp4a_ss(0x01010101u, xa.x, 0);
                            sx = dp4a_ss(0x01010101u, xa.y, sx);
                            sx = dp4a_ss(0x01010101u, xa.z, sx);
                            sx = dp4a_ss(0x01010101u, xa.w, sx);
                            sx = dp4a_ss(0x01010101u, xb.x, sx);
                            sx = dp4a_ss(0x01010101u, xb.y, sx);
                            sx = dp4a_ss(0x01010101u, xb.z, sx);
                            sx = dp4a_ss(0x01010101u, xb.w, sx);
                            s -= 8 * sx;
                            acc[m] = fmaf((float)s, dwf * dxr[m * G + g], acc[m]);
                        }
                    }
                }
            }
        }
    }
    // warp reduction of the binary32 partials (fixed butterfly order)
#pragma unroll
    for (int m = 0; m < M; ++m) {
        float v = acc[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        acc[m] = v;
    }
    if (W == 1) {
        if (lane == 0 && n < N) {
#pragma unroll
            for (int m = 0; m < M; ++m) y[m * ldy + n] = acc[m];
        }
        return;
    }
    if (lane == 0) {
#pragma unroll
        for (int m = 0; m < M; ++m) part[warp][m] = acc[m];
    }
    __syncthreads();
    if (threadIdx.x < R * M) {
        const int r = threadIdx.x / M, m = threadIdx.x % M;
        const int64_t nn = (int64_t)blockIdx.x * R + r;
        if (nn < N) {
            float v = part[r * W][m];
#pragma unroll
            for (int s = 1; s < W; ++s) v += part[r * W + s][m];
            y[m * ldy + nn] = v;
        }
    }
}

template <int M, bool kQ4>
cudaError_t launch_w(int W, const int8_t* qx, const float* dx, const uint8_t* qw,
                     const uint16_t* dw, float* y, int64_t N, int64_t K, int64_t ldy,
                     cudaStream_t s) {
    const int R = kWarps / W;
    const int64_t blocks = (N + R - 1) / R;
    switch (W) {
        case 1: gemv_kernel<M, kQ4, 1><<<blocks, 256, 0, s>>>(qx, dx, qw, dw, y, N, K, ldy); break;
        case 2: gemv_kernel<M, kQ4, 2><<<blocks, 256, 0, s>>>(qx, dx, qw, dw, y, N, K, ldy); break;
        case 4: gemv_kernel<M, kQ4, 4><<<blocks, 256, 0, s>>>(qx, dx, qw, dw, y, N, K, ldy); break;
        default: gemv_kernel<M, kQ4, 8><<<blocks, 256, 0, s>>>(qx, dx, qw, dw, y, N, K, ldy); break;
    }
    return cudaGetLastError();
}

}  // namespace

// K-split factor: enough blocks to fill the GPU a few times over, while each
// warp keeps at least one full 512-byte step of weights.
int gemv_split(int64_t N, int64_t K, bool q4, int sm) {
    const int64_t row_bytes = q4 ? K / 2 : K;
    const int64_t want_blocks = (int64_t)sm * 16;
    int W = 1;
    while (W < 8 && (N * W) / kWarps < want_blocks && row_bytes / (2 * W) >= 512) W *= 2;
    return W;
}

cudaError_t launch_gemv(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                        const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                        cudaStream_t s) {
    const int W = gemv_split(N, K, q4, sm_count());
    const uint8_t* w = (const uint8_t*)qw;
#define QG_GEMV_CASE(MM)                                                              \
    case MM:                                                                          \
        return q4 ? launch_w<MM, true>(W, qx, dx, w, dw, y, N, K, ldy, s)             \
                  : launch_w<MM, false>(W, qx, dx, w, dw, y, N, K, ldy, s);
    switch (M) {
        QG_GEMV_CASE(1) QG_GEMV_CASE(2) QG_GEMV_CASE(3) QG_GEMV_CASE(4)
        QG_GEMV_CASE(5) QG_GEMV_CASE(6) QG_GEMV_CASE(7) QG_GEMV_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef QG_GEMV_CASE
}

}  // namespace qg
