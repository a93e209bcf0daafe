// Decode GEMV (M <= 8): y[m,n] = sum_g dw[n,g] dx[m,g] S[m,n,g] for Q8_0 or
// Q4_0 weights, bound by the weight stream from HBM.
//
// The thin-M product is a structural bandwidth problem ("A 35B
// Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU", Results:
// thin-M GEMM is the limit; Methodology 1: a W4A8 integer decode kernel), so
// the kernel is organised around the weight bytes:
//   * a warp streams R = 4 weight rows over the same K-slice with 16-byte
//     ld.global.nc loads (512 contiguous bytes per row per warp step); the
//     activation bytes of the slice are loaded once per step and reused for
//     the R rows, so activation traffic through L1 is 1/R of the weight bytes
//     per activation row;
//   * group dot products are exact int32 sums of dp4a (Q8: a lane holds half a
//     group and the two halves meet through one shuffle; Q4: a lane holds a
//     whole 16-byte group);
//   * each exact S is scaled by dw * dx and added to a binary32 partial;
//   * split-K: the 8 warps of a block cover (8 / W) row sets x W K-slices;
//     the W binary32 partials of a row meet in shared memory and are summed in
//     slice order, so the result is deterministic for a given shape.  Partial
//     accumulators stay in binary32 (the mining-card page's split-K
//     FlashAttention section: half-precision partials drifted, binary32 ones
//     did not).
// Two kernels implement this:
//   gemv_kernel     one block per row tile, activations read from global
//                   memory (through L1); every shape at M = 1, Q4, and Q8 at
//                   M >= 2 below 8192 rows;
//   gemv_fx_kernel  one resident wave of persistent blocks, each staging the
//                   whole activation (its codes and scales, or the binary32 x
//                   it quantizes itself) in shared memory before walking its
//                   row tiles; Q8 at M >= 2 from 8192 rows takes a whole group
//                   per lane there (8 dp4a, no shuffle).  It also serves
//                   qgemv_q8_0_f32, with the same layout rule, so both entry
//                   points give the same bits.
#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

constexpr int kWarps = 8;

// Q8 at 2 <= M <= 4 with a K-split (W > 1) or M = 2: three resident blocks
// per SM (<= 80 registers a thread, no spills) keep 24 warps' weight loads in
// flight, which the stream needs to cover HBM latency; M = 1 fits three blocks
// unforced.
template <int M, int R, bool kQ4, int W>
__global__ void __launch_bounds__(256, (!kQ4 && M >= 2 && M <= 4 && (W > 1 || M == 2)) ? 3 : 2)
gemv_kernel(const int8_t* __restrict__ qx, const float* __restrict__ dx,
            const uint8_t* __restrict__ qw, const uint16_t* __restrict__ dw,
            float* __restrict__ y, int64_t N, int64_t K, int64_t ldy) {
    constexpr int SETS = kWarps / W;          // row sets per block
    constexpr int U = (R >= 4) ? 1 : 4;       // steps in flight per lane (x R rows)
    __shared__ float part[kWarps][R][M];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = K / kGroup;
    const int64_t n0 = ((int64_t)blockIdx.x * SETS + warp / W) * R;
    const int split = warp % W;
    pdl_wait();                               // x, scales and weights may come from the previous kernel
    float acc[R][M];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

    if (n0 < N) {
        const int64_t gps = (G + W - 1) / W;       // K-slice of this warp, whole groups
        const int64_t g0 = split * gps;
        const int64_t g1 = min64(G, g0 + gps);
        const uint8_t* rowp[R];
        bool rok[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            rok[r] = n0 + r < N;
            rowp[r] = qw + (rok[r] ? n0 + r : n0) * (kQ4 ? K / 2 : K);
        }
        if (!kQ4) {
            // a lane holds 16 bytes = half a group; a step covers 16 groups
            const int64_t b0 = g0 * kGroup, b1 = g1 * kGroup;
            for (int64_t base = b0; base < b1; base += 512 * U) {
                uint4 wv[U][R];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t off = base + u * 512 + lane * 16;
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        wv[u][r] = (off < b1 && rok[r]) ? ldg_nc_v4(rowp[r] + off) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t off = base + u * 512 + lane * 16;
                    const bool ok = off < b1;              // same for both lanes of a group
                    const int64_t g = off / kGroup;
                    float dwf[R];
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        dwf[r] = (ok && rok[r]) ? half_bits_to_float(dw[(n0 + r) * G + g]) : 0.f;
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const uint4 xv = ok ? ldg_v4(qx + m * K + off) : make_uint4(0, 0, 0, 0);
                        const float dxm = ok ? dx[m * G + g] : 0.f;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            int s = dp4a_ss(wv[u][r].x, xv.x, 0);
                            s = dp4a_ss(wv[u][r].y, xv.y, s);
                            s = dp4a_ss(wv[u][r].z, xv.z, s);
                            s = dp4a_ss(wv[u][r].w, xv.w, s);
                            s += __shfl_xor_sync(0xffffffffu, s, 1);   // exact group sum
                            if ((lane & 1) == 0) acc[r][m] = fmaf((float)s, dwf[r] * dxm, acc[r][m]);
                        }
                    }
                }
            }
        } else {
            // a lane holds one whole 16-byte group; a step covers 32 groups
            for (int64_t gb = g0; gb < g1; gb += 32 * U) {
                uint4 wv[U][R];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t g = gb + u * 32 + lane;
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        wv[u][r] = (g < g1 && rok[r]) ? ldg_nc_v4(rowp[r] + g * 16) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t g = gb + u * 32 + lane;
                    if (g < g1) {
                        float dwf[R];
#pragma unroll
                        for (int r = 0; r < R; ++r)
                            dwf[r] = rok[r] ? half_bits_to_float(dw[(n0 + r) * G + g]) : 0.f;
#pragma unroll
                        for (int m = 0; m < M; ++m) {
                            const uint4 xa = ldg_v4(qx + m * K + g * kGroup);
                            const uint4 xb = ldg_v4(qx + m * K + g * kGroup + 16);
                            const float dxm = dx[m * G + g];
                            int sx = dp4a_ss(0x01010101u, xa.x, 0);
                            sx = dp4a_ss(0x01010101u, xa.y, sx);
                            sx = dp4a_ss(0x01010101u, xa.z, sx);
                            sx = dp4a_ss(0x01010101u, xa.w, sx);
                            sx = dp4a_ss(0x01010101u, xb.x, sx);
                            sx = dp4a_ss(0x01010101u, xb.y, sx);
                            sx = dp4a_ss(0x01010101u, xb.z, sx);
                            sx = dp4a_ss(0x01010101u, xb.w, sx);
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                // byte j: element j (low nibble), element j+16 (high)
                                const uint4 w = wv[u][r];
                                int s = dp4a_us(w.x & 0x0f0f0f0fu, xa.x, 0);
                                s = dp4a_us(w.y & 0x0f0f0f0fu, xa.y, s);
                                s = dp4a_us(w.z & 0x0f0f0f0fu, xa.z, s);
                                s = dp4a_us(w.w & 0x0f0f0f0fu, xa.w, s);
                                s = dp4a_us((w.x >> 4) & 0x0f0f0f0fu, xb.x, s);
                                s = dp4a_us((w.y >> 4) & 0x0f0f0f0fu, xb.y, s);
                                s = dp4a_us((w.z >> 4) & 0x0f0f0f0fu, xb.z, s);
                                s = dp4a_us((w.w >> 4) & 0x0f0f0f0fu, xb.w, s);
                                s -= 8 * sx;               // sum (q+8) x - 8 sum x, exact
                                acc[r][m] = fmaf((float)s, dwf[r] * dxm, acc[r][m]);
                            }
                        }
                    }
                }
            }
        }
    }
    // every load of this block is done: the next kernel may start launching
    // (it still waits for this grid to finish before it reads anything)
    pdl_release();
    // warp reduction of the binary32 partials (fixed butterfly order)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float v = acc[r][m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[r][m] = v;
        }
    if (W == 1) {
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (n0 + r < N) {
#pragma unroll
                    for (int m = 0; m < M; ++m) y[m * ldy + n0 + r] = acc[r][m];
                }
        }
        return;
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) part[warp][r][m] = acc[r][m];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < SETS * R * M; i += blockDim.x) {
        const int set = i / (R * M), r = (i / M) % R, m = i % M;
        const int64_t n = ((int64_t)blockIdx.x * SETS + set) * R + r;
        if (n < N) {
            float v = part[set * W][r][m];
#pragma unroll
            for (int s = 1; s < W; ++s) v += part[set * W + s][r][m];
            y[m * ldy + n] = v;
        }
    }
}

// ---- activation quantization fused into the GEMV (binary32 x in) ---------------
//
// y = (Q8 weights) x quant(x) with quant the activation rule of
// quantize_act_q8, bit for bit: one resident wave of persistent blocks, each
// first quantizing all M x K activations into shared memory (8 threads per
// group, max|x| by shuffles, d = max / 127 and every code by IEEE binary32
// division, round-half-even, clamp), then walking row tiles b, b + grid, ...
// with the arithmetic and summation order of gemv_kernel (Q8, 4 rows a warp,
// W K-slices a row set).  One launch instead of two, at the price of every
// block reading and quantizing the whole of x before its first weight load.
__device__ __forceinline__ int quant_code(float v, float d) {
    if (d == 0.0f) return 0;
    const int q = __float2int_rn(__fdiv_rn(v, d));
    return min(max(q, -127), 127);
}

// kPre: the activations arrive quantized (qx int8 [M][K] in x8, dx [M][G] in
// xd) and are only copied into shared memory; else x holds binary32 [M][ldx].
// kWhole: a lane takes a whole group of each row (see gemv_rows_whole); else
// the half-group layout and arithmetic order of gemv_kernel.
template <int M, int R, int W, bool kPre, bool kWhole>
__global__ void __launch_bounds__(256, M == 1 ? 3 : 2)
gemv_fx_kernel(const float* __restrict__ x, int64_t ldx, bool vec_x, const int8_t* __restrict__ x8,
               const float* __restrict__ xd, const uint8_t* __restrict__ qw,
               const uint16_t* __restrict__ dw, float* __restrict__ y, int64_t N, int64_t K,
               int64_t ldy, int64_t tiles) {
    constexpr int SETS = kWarps / W;
    extern __shared__ __align__(16) uint8_t fx_smem[];  // codes [M][K], then scales [M][G]
    __shared__ float part[kWarps][R][M];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = K / kGroup;
    int8_t* sq = reinterpret_cast<int8_t*>(fx_smem);
    float* sd = reinterpret_cast<float*>(fx_smem + ((M * K + 15) & ~(int64_t)15));
    pdl_wait();                               // x and the weights may come from the previous kernel
    if constexpr (kPre) {
        // copy the codes (16 bytes a thread, four loads in flight) and the scales
        const int64_t n16 = M * K / 16;
        for (int64_t i0 = threadIdx.x; i0 < n16; i0 += 4 * (int64_t)blockDim.x) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t i = i0 + u * (int64_t)blockDim.x;
                if (i < n16) v[u] = ldg_v4(x8 + 16 * i);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t i = i0 + u * (int64_t)blockDim.x;
                if (i < n16) reinterpret_cast<uint4*>(sq)[i] = v[u];
            }
        }
        for (int64_t i = threadIdx.x; i < M * G; i += blockDim.x) sd[i] = xd[i];
    } else {
    // quantize: 8 threads per group, 32 groups per pass and U passes' loads in
    // flight together (the full warp runs every pass)
    constexpr int U = 4;
    const int sub = threadIdx.x & 7;
    const int64_t per_pass = blockDim.x / 8;
    for (int64_t base = 0; base < M * G; base += U * per_pass) {
        float4 v[U];
        int64_t grp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            grp[u] = base + u * per_pass + (threadIdx.x >> 3);
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (grp[u] < M * G) {
                const int64_t m = grp[u] / G, g = grp[u] % G;
                const float* p = x + m * ldx + g * kGroup + sub * 4;
                v[u] = vec_x ? *reinterpret_cast<const float4*>(p) : make_float4(p[0], p[1], p[2], p[3]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float a = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            const float d = __fdiv_rn(a, 127.0f);
            if (grp[u] < M * G) {
                // codes [M][K] and scales [M][G] row-major: the flat group index
                const uint32_t packed = (uint32_t)(quant_code(v[u].x, d) & 0xff) |
                                        ((uint32_t)(quant_code(v[u].y, d) & 0xff) << 8) |
                                        ((uint32_t)(quant_code(v[u].z, d) & 0xff) << 16) |
                                        ((uint32_t)(quant_code(v[u].w, d) & 0xff) << 24);
                *reinterpret_cast<uint32_t*>(sq + grp[u] * kGroup + sub * 4) = packed;
                if (sub == 0) sd[grp[u]] = d;
            }
        }
    }
    }
    __syncthreads();
    const int split = warp % W;
    const int64_t gps = (G + W - 1) / W;
    const int64_t g0 = split * gps, g1 = min64(G, g0 + gps);
    const int64_t b0 = g0 * kGroup, b1 = g1 * kGroup;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t n0 = (tile * SETS + warp / W) * R;
        float acc[R][M];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) acc[r][m] = 0.f;
        if (n0 < N) {
            const uint8_t* rowp[R];
            bool rok[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                rok[r] = n0 + r < N;
                rowp[r] = qw + (rok[r] ? n0 + r : n0) * K;
            }
            if constexpr (kWhole) {
                // a lane holds one whole group (32 bytes) of each row, a step covers 32
                // groups: the group sum is 8 dp4a in one lane, with no shuffle
                for (int64_t gb = g0; gb < g1; gb += 32) {
                    const int64_t g = gb + lane;
                    const bool ok = g < g1;
                    uint4 wa[R], wb[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const bool v = ok && rok[r];
                        wa[r] = v ? ldg_nc_v4(rowp[r] + g * kGroup) : make_uint4(0, 0, 0, 0);
                        wb[r] = v ? ldg_nc_v4(rowp[r] + g * kGroup + 16) : make_uint4(0, 0, 0, 0);
                    }
                    float dwf[R];
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        dwf[r] = (ok && rok[r]) ? half_bits_to_float(dw[(n0 + r) * G + g]) : 0.f;
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const uint4 xa = ok ? *reinterpret_cast<const uint4*>(sq + m * K + g * kGroup) : make_uint4(0, 0, 0, 0);
                        const uint4 xb = ok ? *reinterpret_cast<const uint4*>(sq + m * K + g * kGroup + 16) : make_uint4(0, 0, 0, 0);
                        const float dxm = ok ? sd[m * G + g] : 0.f;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            int s = dp4a_ss(wa[r].x, xa.x, 0);
                            s = dp4a_ss(wa[r].y, xa.y, s);
                            s = dp4a_ss(wa[r].z, xa.z, s);
                            s = dp4a_ss(wa[r].w, xa.w, s);
                            s = dp4a_ss(wb[r].x, xb.x, s);
                            s = dp4a_ss(wb[r].y, xb.y, s);
                            s = dp4a_ss(wb[r].z, xb.z, s);
                            s = dp4a_ss(wb[r].w, xb.w, s);       // exact group sum
                            acc[r][m] = fmaf((float)s, dwf[r] * dxm, acc[r][m]);
                        }
                    }
                }
            } else
            for (int64_t base = b0; base < b1; base += 512) {
                const int64_t off = base + lane * 16;
                const bool ok = off < b1;             // same for both lanes of a group
                uint4 wv[R];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    wv[r] = (ok && rok[r]) ? ldg_nc_v4(rowp[r] + off) : make_uint4(0, 0, 0, 0);
                const int64_t g = off / kGroup;
                float dwf[R];
#pragma unroll
                for (int r = 0; r < R; ++r) dwf[r] = (ok && rok[r]) ? half_bits_to_float(dw[(n0 + r) * G + g]) : 0.f;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const uint4 xv = ok ? *reinterpret_cast<const uint4*>(sq + m * K + off) : make_uint4(0, 0, 0, 0);
                    const float dxm = ok ? sd[m * G + g] : 0.f;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        int s = dp4a_ss(wv[r].x, xv.x, 0);
                        s = dp4a_ss(wv[r].y, xv.y, s);
                        s = dp4a_ss(wv[r].z, xv.z, s);
                        s = dp4a_ss(wv[r].w, xv.w, s);
                        s += __shfl_xor_sync(0xffffffffu, s, 1);   // exact group sum
                        if ((lane & 1) == 0) acc[r][m] = fmaf((float)s, dwf[r] * dxm, acc[r][m]);
                    }
                }
            }
        }
        if (tile + gridDim.x >= tiles) pdl_release();   // this block's last weight loads are issued
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float v = acc[r][m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[r][m] = v;
            }
        if (W == 1) {
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    if (n0 + r < N) {
#pragma unroll
                        for (int m = 0; m < M; ++m) y[m * ldy + n0 + r] = acc[r][m];
                    }
            }
            continue;
        }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < M; ++m) part[warp][r][m] = acc[r][m];
        }
        __syncthreads();
        for (int i = threadIdx.x; i < SETS * R * M; i += blockDim.x) {
            const int set = i / (R * M), r = (i / M) % R, m = i % M;
            const int64_t n = (tile * SETS + set) * R + r;
            if (n < N) {
                float v = part[set * W][r][m];
#pragma unroll
                for (int s = 1; s < W; ++s) v += part[set * W + s][r][m];
                y[m * ldy + n] = v;
            }
        }
        __syncthreads();                      // part is written again for the next tile
    }
}

constexpr size_t kFxSmemMax = 200 * 1024;     // codes + scales of x in one block

template <int M, int R, int W, bool kPre, bool kWhole>
cudaError_t launch_fx_w(const float* x, int64_t ldx, const int8_t* x8, const float* xd,
                        const uint8_t* qw, const uint16_t* dw, float* y, int64_t N, int64_t K,
                        int64_t ldy, cudaStream_t s) {
    auto kern = gemv_fx_kernel<M, R, W, kPre, kWhole>;
    const size_t smem = (size_t)(((M * K + 15) & ~(int64_t)15) + 4 * M * (K / kGroup));
    if (smem > kFxSmemMax) return cudaErrorInvalidValue;
    static const cudaError_t attr =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFxSmemMax);
    if (attr != cudaSuccess) return attr;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem);
    if (e != cudaSuccess) return e;
    const int64_t rows_per_block = (kWarps / W) * R;
    const int64_t tiles = (N + rows_per_block - 1) / rows_per_block;
    int64_t grid = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
    if (grid > tiles) grid = tiles;
    const bool vec_x = ((uintptr_t)x & 15u) == 0 && ldx % 4 == 0;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(256), smem, s, x, ldx, vec_x, x8, xd, qw, dw, y,
                      N, K, ldy, tiles);
}

template <int M, int R, bool kQ4>
cudaError_t launch_w(int W, const int8_t* qx, const float* dx, const uint8_t* qw,
                     const uint16_t* dw, float* y, int64_t N, int64_t K, int64_t ldy,
                     cudaStream_t s) {
    const int rows_per_block = (kWarps / W) * R;
    const int64_t blocks = (N + rows_per_block - 1) / rows_per_block;
    // programmatic launch: the blocks may be scheduled while the previous
    // kernel drains and wait for it in pdl_wait()
    const dim3 g((unsigned)blocks), b(256);
    switch (W) {
        case 1: return launch_pdl(gemv_kernel<M, R, kQ4, 1>, g, b, 0, s, qx, dx, qw, dw, y, N, K, ldy);
        case 2: return launch_pdl(gemv_kernel<M, R, kQ4, 2>, g, b, 0, s, qx, dx, qw, dw, y, N, K, ldy);
        case 4: return launch_pdl(gemv_kernel<M, R, kQ4, 4>, g, b, 0, s, qx, dx, qw, dw, y, N, K, ldy);
        default: return launch_pdl(gemv_kernel<M, R, kQ4, 8>, g, b, 0, s, qx, dx, qw, dw, y, N, K, ldy);
    }
}

// 4 rows per warp, one 512-byte step per row in flight per iteration: at
// M = 1 this beat 2 rows x 4 steps on every decode shape measured (the
// activation loads are shared by more rows and fewer registers are live).
constexpr int rows_per_warp(int M) { (void)M; return 4; }

}  // namespace

// K-split factor: enough blocks to fill the GPU a few times over, while each
// warp keeps at least one full 512-byte step of weights per row.
int gemv_split(int64_t M, int64_t N, int64_t K, bool q4, int sm, int R) {
    const int64_t row_bytes = q4 ? K / 2 : K;
    const int64_t want_blocks = (int64_t)sm * 8;
    // at M >= 2 the split starts at 2: the W = 1 kernel needs more registers
    // than three resident blocks allow
    int W = (M >= 2 && !q4 && row_bytes / 4 >= 512) ? 2 : 1;
    while (W < 8 && (N * W) / (kWarps * R) < want_blocks && row_bytes / (2 * W) >= 512) W *= 2;
    return W;
}

namespace {

// Whether a Q8 product takes a whole group per lane: M >= 2 and at least 8192
// rows (fewer do not amortize each block's staging of the activations: 4096 x
// 4096 and 4096 x 12288 at M = 4 ran 1-3 us slower).  The two-launch path and
// the GEMV that quantizes its own activations follow the same rule, so their
// results stay bit-identical.
bool gemv_rows_whole(int64_t M, int64_t N) { return M >= 2 && N >= 8192; }

// Q8 at M >= 2 on large N: the persistent kernel that stages the quantized
// activations once per block in shared memory and takes a whole group per lane
// (gemv_fx_kernel with kPre).  At M >= 2 the register-fed kernel below is bound
// by instruction issue (the half-group shuffles and the activation loads of
// every step); the M = 4 lm-head ran 155 -> 135 us this way.
template <int MM, int R>
cudaError_t launch_pre(int W, const int8_t* qx, const float* dx, const uint8_t* w, const uint16_t* dw,
                       float* y, int64_t N, int64_t K, int64_t ldy, cudaStream_t s) {
    switch (W) {
        case 1: return launch_fx_w<MM, R, 1, true, true>(nullptr, 0, qx, dx, w, dw, y, N, K, ldy, s);
        case 2: return launch_fx_w<MM, R, 2, true, true>(nullptr, 0, qx, dx, w, dw, y, N, K, ldy, s);
        case 4: return launch_fx_w<MM, R, 4, true, true>(nullptr, 0, qx, dx, w, dw, y, N, K, ldy, s);
        default: return launch_fx_w<MM, R, 8, true, true>(nullptr, 0, qx, dx, w, dw, y, N, K, ldy, s);
    }
}

}  // namespace

cudaError_t launch_gemv(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                        const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                        cudaStream_t s) {
    const uint8_t* w = (const uint8_t*)qw;
    const int sm = sm_count();
    const bool staged = !q4 && gemv_rows_whole(M, N) && (size_t)(M * K + M * K / 8) <= kFxSmemMax;
#define QG_GEMV_CASE(MM)                                                                        \
    case MM: {                                                                                  \
        constexpr int R = rows_per_warp(MM);                                                    \
        const int W = gemv_split(MM, N, K, q4, sm, R);                                          \
        if constexpr (MM >= 2) {                                                                \
            if (staged) return launch_pre<MM, R>(W, qx, dx, w, dw, y, N, K, ldy, s);            \
        }                                                                                       \
        return q4 ? launch_w<MM, R, true>(W, qx, dx, w, dw, y, N, K, ldy, s)                    \
                  : launch_w<MM, R, false>(W, qx, dx, w, dw, y, N, K, ldy, s);                  \
    }
    switch (M) {
        QG_GEMV_CASE(1) QG_GEMV_CASE(2) QG_GEMV_CASE(3) QG_GEMV_CASE(4)
        QG_GEMV_CASE(5) QG_GEMV_CASE(6) QG_GEMV_CASE(7) QG_GEMV_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef QG_GEMV_CASE
}

namespace {

template <int MM, int R, int W>
cudaError_t launch_fx(bool whole, const float* x, int64_t ldx, const uint8_t* w, const uint16_t* dw,
                      float* y, int64_t N, int64_t K, int64_t ldy, cudaStream_t s) {
    if constexpr (MM >= 2) {
        if (whole) return launch_fx_w<MM, R, W, false, true>(x, ldx, nullptr, nullptr, w, dw, y, N, K, ldy, s);
    }
    return launch_fx_w<MM, R, W, false, false>(x, ldx, nullptr, nullptr, w, dw, y, N, K, ldy, s);
}

}  // namespace

cudaError_t launch_gemv_fx(const float* x, int64_t ldx, int64_t M, int64_t N, int64_t K, const void* qw,
                           const uint16_t* dw, float* y, int64_t ldy, cudaStream_t s) {
    const uint8_t* w = (const uint8_t*)qw;
    const int sm = sm_count();
    const bool whole = gemv_rows_whole(M, N);
#define QG_FX_CASE(MM)                                                                          \
    case MM: {                                                                                  \
        constexpr int R = rows_per_warp(MM);                                                    \
        switch (gemv_split(MM, N, K, false, sm, R)) {                                           \
            case 1: return launch_fx<MM, R, 1>(whole, x, ldx, w, dw, y, N, K, ldy, s);           \
            case 2: return launch_fx<MM, R, 2>(whole, x, ldx, w, dw, y, N, K, ldy, s);           \
            case 4: return launch_fx<MM, R, 4>(whole, x, ldx, w, dw, y, N, K, ldy, s);           \
            default: return launch_fx<MM, R, 8>(whole, x, ldx, w, dw, y, N, K, ldy, s);          \
        }                                                                                       \
    }
    switch (M) {
        QG_FX_CASE(1) QG_FX_CASE(2) QG_FX_CASE(3) QG_FX_CASE(4)
        QG_FX_CASE(5) QG_FX_CASE(6) QG_FX_CASE(7) QG_FX_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef QG_FX_CASE
}

}  // namespace qg
