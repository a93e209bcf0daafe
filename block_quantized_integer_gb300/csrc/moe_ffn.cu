// The MoE steps on either side of the grouped GEMM ("A 35B Hybrid-Attention
// Mixture-of-Experts Model on a 6GB 2011 GPU", Methodology 1: grouped 4-bit
// GEMM for MoE routing, 8-bit activations into the W4A8 products;
// Methodology 2: router-weighted experts):
//
//   swiglu_quant: h[p, j] = silu(gate[p, j]) * up[p, j],  silu(v) = v / (1 + e^-v),
//                 then h re-quantized to int8 codes + binary32 scale per
//                 32-group with the activation rule (d = max|h| / 127 by one
//                 IEEE division, q = clamp(round_half_even(h / d), -127, 127)),
//                 ready to be the activation rows of the down projection.
//                 Both quotients are taken as a product with a correctly
//                 rounded binary32 reciprocal (silu: v * rcp(1 + e^-v); codes:
//                 h * rcp(d)): each differs from the IEEE quotient by at most
//                 one rounding, so a code can differ from round_half_even(h / d)
//                 only where h / d lies within ~2^-22 relative of a half-integer;
//   combine:      out[t, n] = sum_{s < topk} w[t, s] * y[t * topk + s, n], the
//                 slots summed in order with binary32 FMAs.
//
// Both are HBM-bound streaming kernels: swiglu_quant reads 8 bytes and writes
// 1.125 per output element; combine reads topk * (4 + 4 / N) bytes and writes
// 4 per output element.
#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fmul_rn(__fmul_rn(g, __frcp_rn(__fadd_rn(1.0f, expf(-g)))), u);
}

// rd = rcp(d) (0 when d == 0: every code of an all-zero group is 0)
__device__ __forceinline__ int quant127(float v, float rd) {
    const int q = __float2int_rn(__fmul_rn(v, rd));
    return min(max(q, -127), 127);
}

// 8 threads per 32-group, 4 consecutive elements (one 16-byte load of gate
// and one of up) per thread; a warp covers 4 groups; U groups per thread have
// their loads in flight together.
template <bool kFast>
__global__ void __launch_bounds__(256)
swiglu_quant_kernel(const float* __restrict__ gu, int64_t P, int64_t F, int64_t ldgu,
                    int8_t* __restrict__ qh, float* __restrict__ dh, bool vec_ok, FastDiv fg) {
    pdl_wait();                               // gu comes from the gate/up GEMM
    pdl_release();
    constexpr int U = 2;
    const int64_t G = F / kGroup;
    const int64_t total = P * G;
    const int sub = threadIdx.x & 7;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 3);
    const int64_t first = (int64_t)blockIdx.x * (blockDim.x >> 3) + (threadIdx.x >> 3);
    const int64_t warp_first = first - ((threadIdx.x & 31) >> 3);
    for (int64_t base = warp_first; base < total; base += U * stride) {   // whole warps iterate
        float4 a[U], b[U];
        int64_t grp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            grp[u] = base + u * stride + ((threadIdx.x & 31) >> 3);
            a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (grp[u] < total) {
                int64_t pr, g;
                if constexpr (kFast) {
                    pr = fg.div((uint32_t)grp[u]);
                    g = grp[u] - pr * G;
                } else {
                    pr = grp[u] / G;
                    g = grp[u] % G;
                }
                const float* gp = gu + pr * ldgu + g * kGroup + sub * 4;
                if (vec_ok) {
                    a[u] = *reinterpret_cast<const float4*>(gp);
                    b[u] = *reinterpret_cast<const float4*>(gp + F);
                } else {
                    a[u] = make_float4(gp[0], gp[1], gp[2], gp[3]);
                    b[u] = make_float4(gp[F], gp[F + 1], gp[F + 2], gp[F + 3]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool active = grp[u] < total;
            float h[4] = {0.f, 0.f, 0.f, 0.f};
            if (active) {
                h[0] = silu_mul(a[u].x, b[u].x);
                h[1] = silu_mul(a[u].y, b[u].y);
                h[2] = silu_mul(a[u].z, b[u].z);
                h[3] = silu_mul(a[u].w, b[u].w);
            }
            float m = fmaxf(fmaxf(fabsf(h[0]), fabsf(h[1])), fmaxf(fabsf(h[2]), fabsf(h[3])));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            const float d = __fdiv_rn(m, 127.0f);
            const float rd = d == 0.0f ? 0.0f : __frcp_rn(d);
            if (active) {
                const uint32_t packed = (uint32_t)(quant127(h[0], rd) & 0xff) |
                                        ((uint32_t)(quant127(h[1], rd) & 0xff) << 8) |
                                        ((uint32_t)(quant127(h[2], rd) & 0xff) << 16) |
                                        ((uint32_t)(quant127(h[3], rd) & 0xff) << 24);
                // [P][F] codes and [P][G] scales at the flat group index
                *reinterpret_cast<uint32_t*>(qh + grp[u] * kGroup + sub * 4) = packed;
                if (sub == 0) dh[grp[u]] = d;
            }
        }
    }
}

// One thread per 4 consecutive outputs of a token row (vec) or per output.
constexpr int kSlots = 8;
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ y, const float* __restrict__ w, int64_t T, int topk,
               int64_t N, float* __restrict__ out, bool vec4) {
    pdl_wait();                               // y comes from the down GEMM
    pdl_release();
    const int64_t per_row = vec4 ? N / 4 : N;
    const int64_t total = T * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_row, c = i % per_row;
        const float* wt = w + t * topk;
        const float* yt = y + t * topk * N;
        if (vec4) {
            // the first kSlots slots' loads all go out before the first FMA;
            // the sum still runs over the slots in order
            float4 v[kSlots];
            float ws[kSlots];
#pragma unroll
            for (int s = 0; s < kSlots; ++s)
                if (s < topk) {
                    ws[s] = wt[s];
                    v[s] = *reinterpret_cast<const float4*>(yt + s * N + 4 * c);
                }
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int s = 0; s < kSlots; ++s)
                if (s < topk) {
                    acc.x = fmaf(ws[s], v[s].x, acc.x);
                    acc.y = fmaf(ws[s], v[s].y, acc.y);
                    acc.z = fmaf(ws[s], v[s].z, acc.z);
                    acc.w = fmaf(ws[s], v[s].w, acc.w);
                }
            for (int s = kSlots; s < topk; ++s) {
                const float w1 = wt[s];
                const float4 v1 = *reinterpret_cast<const float4*>(yt + s * N + 4 * c);
                acc.x = fmaf(w1, v1.x, acc.x);
                acc.y = fmaf(w1, v1.y, acc.y);
                acc.z = fmaf(w1, v1.z, acc.z);
                acc.w = fmaf(w1, v1.w, acc.w);
            }
            *reinterpret_cast<float4*>(out + t * N + 4 * c) = acc;
        } else {
            float acc = 0.f;
            for (int s = 0; s < topk; ++s) acc = fmaf(wt[s], yt[s * N + c], acc);
            out[t * N + c] = acc;
        }
    }
}

int stream_grid(int64_t work) {
    int64_t b = (work + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_swiglu_quant(const float* gu, int64_t P, int64_t F, int64_t ldgu, int8_t* qh,
                                float* dh, cudaStream_t s) {
    const bool vec_ok = ((uintptr_t)gu % 16 == 0) && (ldgu % 4 == 0) && (F % 4 == 0);
    const int64_t total = P * (F / kGroup);
    const dim3 grid(stream_grid(total * 8)), block(256);
    if (total < (1ll << 32))
        return launch_pdl(swiglu_quant_kernel<true>, grid, block, 0, s, gu, P, F, ldgu, qh, dh, vec_ok,
                          FastDiv((uint32_t)(F / kGroup)));
    return launch_pdl(swiglu_quant_kernel<false>, grid, block, 0, s, gu, P, F, ldgu, qh, dh, vec_ok,
                      FastDiv(1));
}

cudaError_t launch_combine(const float* y, const float* w, int64_t T, int topk, int64_t N,
                           float* out, cudaStream_t s) {
    const bool vec4 = (N % 4 == 0) && ((uintptr_t)y % 16 == 0) && ((uintptr_t)out % 16 == 0);
    return launch_pdl(combine_kernel, dim3(stream_grid(T * (vec4 ? N / 4 : N))), dim3(256), 0, s, y, w, T,
                      topk, N, out, vec4);
}

}  // namespace qg
