// Group quantizers: activations (int8, binary32 scale) and weights (Q8_0 /
// Q4_0, binary16 scale), 32 elements per group along K.
//
// Rule (Q8 block format of "I wrote a custom CUDA inference engine to run
// Qwen3.5-27B on a $130 mining card", Features; 8-bit activations and
// group-wise symmetric 4-bit weights of "A 35B Hybrid-Attention
// Mixture-of-Experts Model on a 6GB 2011 GPU", Methodology 2):
//   d = max|v| / qmax by one IEEE binary32 division (__fdiv_rn),
//   weights: d rounded to binary16 (nearest-even, saturated to 65504) first,
//   q = clamp(round_half_even(v / d), lo, hi) with a binary32 quotient,
//   d == 0 gives q = 0.
// Built without --use_fast_math and without flush-to-zero, so subnormal
// scales divide exactly as IEEE says.
//
// Layout of the work: activations 4 threads per group with 8 consecutive
// elements each (two 16-byte loads, a warp covers 8 groups = 1 KiB of input);
// weights 8 threads per group with 4 elements each (one 16-byte load).
// HBM-bound: 4 bytes read and 1.125 (activations) / 1.0625 (Q8) / 0.5625 (Q4)
// bytes written per element.
#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

__device__ __forceinline__ float amax8(float a) {
    // max over the 8 lanes of one group (lanes 8j .. 8j+7)
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    return a;
}

__device__ __forceinline__ int quant1(float v, float d, int lo, int hi) {
    if (d == 0.0f) return 0;
    int q = __float2int_rn(__fdiv_rn(v, d));
    return min(max(q, lo), hi);
}

__device__ __forceinline__ float4 load4(const float* p, bool vec_ok) {
    if (vec_ok) return *reinterpret_cast<const float4*>(p);
    return make_float4(p[0], p[1], p[2], p[3]);
}

__device__ __forceinline__ uint32_t pack_s8(int a, int b, int c, int d) {
    return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) |
           ((uint32_t)(c & 0xff) << 16) | ((uint32_t)(d & 0xff) << 24);
}

// binary16 scale from max|v| / qmax, saturated at the largest finite value.
__device__ __forceinline__ uint16_t scale16(float amax, float qmax) {
    __half h = __float2half_rn(__fdiv_rn(amax, qmax));
    uint16_t b = __half_as_ushort(h);
    if ((b & 0x7fffu) == 0x7c00u) b = (uint16_t)((b & 0x8000u) | 0x7bffu);
    return b;
}

// kFast: M * G < 2^32, flat group index split into (row, group) by FastDiv.
// 4 threads per group, 8 consecutive elements (two 16-byte loads) per thread,
// U groups per thread with their loads in flight together; a warp covers 8
// groups = 1 KiB of contiguous input per pass.
template <bool kFast>
__global__ void __launch_bounds__(256)
quantize_act_q8_kernel(const float* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                       int8_t* __restrict__ qx, float* __restrict__ dx, bool vec_ok, FastDiv fg) {
    constexpr int U = 2;                          // groups per thread in flight
    const int64_t G = K / kGroup;
    const int64_t total = M * G;
    const int sub = threadIdx.x & 3;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 2);
    // Every lane of a warp runs the same number of iterations (the shuffles
    // need the full warp), so the loop bound is rounded up to whole warps.
    const int64_t first = (int64_t)blockIdx.x * (blockDim.x >> 2) + (threadIdx.x >> 2);
    const int64_t warp_first = first - ((threadIdx.x & 31) >> 2);
    pdl_wait();                               // x may come from the previous kernel
    pdl_release();                            // the next kernel may launch and wait for this one
    for (int64_t base = warp_first; base < total; base += U * stride) {
        float4 v[U][2];
        int64_t grp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {             // all loads first
            grp[u] = base + u * stride + ((threadIdx.x & 31) >> 2);
            v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (grp[u] < total) {
                int64_t m, g;
                if constexpr (kFast) {
                    m = fg.div((uint32_t)grp[u]);
                    g = grp[u] - m * G;
                } else {
                    m = grp[u] / G;
                    g = grp[u] % G;
                }
                const float* p = x + m * ldx + g * kGroup + sub * 8;
                v[u][0] = load4(p, vec_ok);
                v[u][1] = load4(p + 4, vec_ok);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool active = grp[u] < total;
            float a = fmaxf(fmaxf(fmaxf(fabsf(v[u][0].x), fabsf(v[u][0].y)), fmaxf(fabsf(v[u][0].z), fabsf(v[u][0].w))),
                            fmaxf(fmaxf(fabsf(v[u][1].x), fabsf(v[u][1].y)), fmaxf(fabsf(v[u][1].z), fabsf(v[u][1].w))));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));    // max over the group's 4 lanes
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            const float d = __fdiv_rn(a, 127.0f);
            if (active) {
                // codes and scales are stored at the flat group index: [M][G] row-major
                const uint32_t lo = pack_s8(quant1(v[u][0].x, d, -127, 127), quant1(v[u][0].y, d, -127, 127),
                                            quant1(v[u][0].z, d, -127, 127), quant1(v[u][0].w, d, -127, 127));
                const uint32_t hi = pack_s8(quant1(v[u][1].x, d, -127, 127), quant1(v[u][1].y, d, -127, 127),
                                            quant1(v[u][1].z, d, -127, 127), quant1(v[u][1].w, d, -127, 127));
                *reinterpret_cast<uint2*>(qx + grp[u] * kGroup + sub * 8) = make_uint2(lo, hi);
                if (sub == 0) dx[grp[u]] = d;
            }
        }
    }
}

template <bool kQ4>
__global__ void __launch_bounds__(256)
quantize_weight_kernel(const float* __restrict__ w, int64_t N, int64_t K,
                       uint8_t* __restrict__ qw, uint16_t* __restrict__ dw, bool vec_ok) {
    const int64_t G = K / kGroup;
    const int64_t total = N * G;
    const int sub = threadIdx.x & 7;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 3);
    const int64_t first = (int64_t)blockIdx.x * (blockDim.x >> 3) + (threadIdx.x >> 3);
    const int64_t warp_first = first - ((threadIdx.x & 31) >> 3);
    const float qmax = kQ4 ? 7.0f : 127.0f;
    const int lo = kQ4 ? -8 : -127, hi = kQ4 ? 7 : 127;
    for (int64_t base = warp_first; base < total; base += stride) {
        const int64_t grp = base + ((threadIdx.x & 31) >> 3);
        const bool active = grp < total;
        const int64_t n = active ? grp / G : 0, g = active ? grp % G : 0;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active) v = load4(w + n * K + g * kGroup + sub * 4, vec_ok);
        float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        a = amax8(a);
        const uint16_t h = scale16(a, qmax);
        const float d = half_bits_to_float(h);
        int q0 = quant1(v.x, d, lo, hi), q1 = quant1(v.y, d, lo, hi);
        int q2 = quant1(v.z, d, lo, hi), q3 = quant1(v.w, d, lo, hi);
        if (!kQ4) {
            if (active) {
                *reinterpret_cast<uint32_t*>(qw + n * K + g * kGroup + sub * 4) =
                    pack_s8(q0, q1, q2, q3);
                if (sub == 0) dw[n * G + g] = h;
            }
        } else {
            // Thread sub (0..3) holds elements 4sub..4sub+3 (low nibbles of
            // bytes 4sub..4sub+3); thread sub+4 holds elements 16+4sub.. (the
            // high nibbles of the same bytes).
            uint32_t lo_n = (uint32_t)(q0 + 8) | ((uint32_t)(q1 + 8) << 8) |
                            ((uint32_t)(q2 + 8) << 16) | ((uint32_t)(q3 + 8) << 24);
            uint32_t hi_n = __shfl_down_sync(0xffffffffu, lo_n, 4);
            if (active && sub < 4) {
                *reinterpret_cast<uint32_t*>(qw + n * (K / 2) + g * (kGroup / 2) + sub * 4) =
                    lo_n | (hi_n << 4);
                if (sub == 0) dw[n * G + g] = h;
            }
        }
    }
}

int grid_for(int64_t groups, int sm_count) {
    int64_t need = (groups + 31) / 32;          // 32 groups per 256-thread block
    int64_t cap = (int64_t)sm_count * 8 * 4;    // a few waves of resident blocks
    if (need > cap) need = cap;
    return (int)(need < 1 ? 1 : need);
}

}  // namespace

cudaError_t launch_quantize_act_q8(const float* x, int64_t M, int64_t K, int64_t ldx,
                                   int8_t* qx, float* dx, cudaStream_t s) {
    const bool vec_ok = ((uintptr_t)x % 16 == 0) && (ldx % 4 == 0);
    const int64_t total = M * (K / kGroup);
    const dim3 grid(grid_for(total, sm_count())), block(256);
    if (total < (1ll << 32))
        return launch_pdl(quantize_act_q8_kernel<true>, grid, block, 0, s, x, M, K, ldx, qx, dx, vec_ok,
                          FastDiv((uint32_t)(K / kGroup)));
    return launch_pdl(quantize_act_q8_kernel<false>, grid, block, 0, s, x, M, K, ldx, qx, dx, vec_ok,
                      FastDiv(1));
}

cudaError_t launch_quantize_weight(const float* w, int64_t N, int64_t K, void* qw,
                                   uint16_t* dw, bool q4, cudaStream_t s) {
    const bool vec_ok = ((uintptr_t)w % 16 == 0);
    const int grid = grid_for(N * (K / kGroup), sm_count());
    if (q4)
        quantize_weight_kernel<true><<<grid, 256, 0, s>>>(w, N, K, (uint8_t*)qw, dw, vec_ok);
    else
        quantize_weight_kernel<false><<<grid, 256, 0, s>>>(w, N, K, (uint8_t*)qw, dw, vec_ok);
    return cudaGetLastError();
}

}  // namespace qg
