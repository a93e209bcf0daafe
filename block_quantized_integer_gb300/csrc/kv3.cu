// 3-bit KV-cache codec: Walsh-Hadamard rotation + Lloyd-Max scalar quantizer
// ("I wrote a custom CUDA inference engine to run Qwen3.5-27B on a $130
// mining card", Features: a 3-bit Walsh-Hadamard + Lloyd-Max KV cache that
// fits a 256 K context; the second page about the same engine: 17 GB of KV
// cache down to 3.5 GB).  The pages name the two steps only; the reading
// taken here:
//   * a vector is one head's D values (D = 64, 128 or 256);
//   * y = H x / sqrt(D) with H the Sylvester-ordered Hadamard matrix
//     (orthonormal, its own inverse);
//   * s = sqrt(mean(y^2)) in binary32, stored per vector;
//   * each y_j / s is coded as the index (0..7) of the nearest of the 8
//     Lloyd-Max reconstruction levels of the standard normal distribution
//     (the optimal 3-bit quantizer for a unit Gaussian; the rotation makes the
//     coefficients close to Gaussian): code = number of decision thresholds
//     <= y_j / s, with the thresholds halfway between adjacent levels;
//   * the codes of a vector are stored as 3 bit planes of D bits: word
//     b * (D/32) + e, bit L holds bit b of the code of element L * (D/32) + e;
//   * decode: x^ = H (s * level[code]) / sqrt(D).
// A vector takes 3 D / 8 + 4 bytes (52 for D = 128) instead of 2 D in
// binary16: 4.9 times smaller.
//
// The codebook is computed on the host from its defining conditions (each
// level the mean of the normal distribution over its cell, each threshold the
// midpoint of its two levels) by Lloyd's iteration in binary64 and rounded to
// binary32 once.  One warp per vector: lane L holds elements L*E .. L*E+E-1
// (E = D / 32); butterflies below E run inside a lane, the others through
// shuffles.  HBM-bound: 4 D bytes in and 3 D / 8 + 4 out per vector (encode).
#include <math.h>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

struct Codebook {
    float level[8];
    float thr[7];
};

// Lloyd's iteration for the 8-level quantizer of N(0, 1), binary64.
Codebook make_codebook() {
    const double kInvSqrt2Pi = 0.39894228040143267794;
    auto pdf = [&](double t) { return isinf(t) ? 0.0 : kInvSqrt2Pi * exp(-0.5 * t * t); };
    auto cdf = [](double t) { return 0.5 * erfc(-t / sqrt(2.0)); };
    double lv[8], th[9];
    for (int k = 0; k < 8; ++k) lv[k] = -1.75 + 0.5 * k;
    for (int it = 0; it < 5000; ++it) {
        th[0] = -INFINITY;
        th[8] = INFINITY;
        for (int k = 1; k < 8; ++k) th[k] = 0.5 * (lv[k - 1] + lv[k]);
        double change = 0.0;
        for (int k = 0; k < 8; ++k) {
            const double mass = cdf(th[k + 1]) - cdf(th[k]);
            const double c = (pdf(th[k]) - pdf(th[k + 1])) / mass;
            change = fmax(change, fabs(c - lv[k]));
            lv[k] = c;
        }
        if (change < 1e-16) break;
    }
    Codebook cb;
    for (int k = 0; k < 8; ++k) cb.level[k] = (float)lv[k];
    for (int k = 0; k < 7; ++k) cb.thr[k] = (float)(0.5 * (lv[k] + lv[k + 1]));
    return cb;
}

const Codebook& codebook() {
    static Codebook cb;
    static std::once_flag once;
    std::call_once(once, [] { cb = make_codebook(); });
    return cb;
}

// In-warp orthonormal Walsh-Hadamard transform of D = 32 E values; r is
// 1 / sqrt(D) rounded to binary32 once (on the host, in binary64).
template <int E>
__device__ __forceinline__ void wht_warp(float (&v)[E], int lane, float r) {
#pragma unroll
    for (int h = 1; h < E; h <<= 1)
#pragma unroll
        for (int e = 0; e < E; ++e)
            if ((e & h) == 0) {
                const float a = v[e], b = v[e + h];
                v[e] = a + b;
                v[e + h] = a - b;
            }
#pragma unroll
    for (int hl = 1; hl < 32; hl <<= 1)
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float p = __shfl_xor_sync(0xffffffffu, v[e], hl);
            v[e] = (lane & hl) ? p - v[e] : v[e] + p;
        }
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] *= r;
}

template <int E>
__global__ void __launch_bounds__(256)
kv3_encode_kernel(const float* __restrict__ x, int64_t T, int64_t ldx, uint32_t* __restrict__ codes,
                  float* __restrict__ scales, Codebook cb, float r) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        float v[E];
        const float* xr = x + t * ldx + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = xr[e];
        wht_warp<E>(v, lane, r);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float s = sqrtf(__fdiv_rn(ss, (float)(32 * E)));
        uint32_t c[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            uint32_t k = 0;
            if (s > 0.f) {
                const float u = __fdiv_rn(v[e], s);
#pragma unroll
                for (int i = 0; i < 7; ++i) k += (u >= cb.thr[i]) ? 1u : 0u;
            }
            c[e] = k;
        }
        uint32_t* out = codes + t * (3 * E);
#pragma unroll
        for (int b = 0; b < 3; ++b)
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const uint32_t w = __ballot_sync(0xffffffffu, (c[e] >> b) & 1u);
                if (lane == 0) out[b * E + e] = w;
            }
        if (lane == 0) scales[t] = s;
    }
}

template <int E>
__global__ void __launch_bounds__(256)
kv3_decode_kernel(const uint32_t* __restrict__ codes, const float* __restrict__ scales, int64_t T,
                  float* __restrict__ x, int64_t ldx, Codebook cb, float r) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        const uint32_t* in = codes + t * (3 * E);
        const uint32_t mine = lane < 3 * E ? in[lane] : 0u;     // one word per lane, then shuffled
        const float s = scales[t];
        float v[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const uint32_t w0 = __shfl_sync(0xffffffffu, mine, e);
            const uint32_t w1 = __shfl_sync(0xffffffffu, mine, E + e);
            const uint32_t w2 = __shfl_sync(0xffffffffu, mine, 2 * E + e);
            const uint32_t k = ((w0 >> lane) & 1u) | (((w1 >> lane) & 1u) << 1) | (((w2 >> lane) & 1u) << 2);
            float lvl = cb.level[0];
#pragma unroll
            for (int i = 1; i < 8; ++i) lvl = (k == (uint32_t)i) ? cb.level[i] : lvl;
            v[e] = s * lvl;
        }
        wht_warp<E>(v, lane, r);
        float* xr = x + t * ldx + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) xr[e] = v[e];
    }
}

int grid_vectors(int64_t T) {
    int64_t b = (T + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace

void kv3_codebook(float* levels, float* thresholds) {
    const Codebook& cb = codebook();
    for (int k = 0; k < 8; ++k) levels[k] = cb.level[k];
    for (int k = 0; k < 7; ++k) thresholds[k] = cb.thr[k];
}

cudaError_t launch_kv3_encode(const float* x, int64_t T, int D, int64_t ldx, uint32_t* codes,
                              float* scales, cudaStream_t s) {
    const Codebook& cb = codebook();
    const int g = grid_vectors(T);
    const float r = (float)(1.0 / sqrt((double)D));
    switch (D) {
        case 64: kv3_encode_kernel<2><<<g, 256, 0, s>>>(x, T, ldx, codes, scales, cb, r); break;
        case 128: kv3_encode_kernel<4><<<g, 256, 0, s>>>(x, T, ldx, codes, scales, cb, r); break;
        case 256: kv3_encode_kernel<8><<<g, 256, 0, s>>>(x, T, ldx, codes, scales, cb, r); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_kv3_decode(const uint32_t* codes, const float* scales, int64_t T, int D,
                              float* x, int64_t ldx, cudaStream_t s) {
    const Codebook& cb = codebook();
    const int g = grid_vectors(T);
    const float r = (float)(1.0 / sqrt((double)D));
    switch (D) {
        case 64: kv3_decode_kernel<2><<<g, 256, 0, s>>>(codes, scales, T, x, ldx, cb, r); break;
        case 128: kv3_decode_kernel<4><<<g, 256, 0, s>>>(codes, scales, T, x, ldx, cb, r); break;
        case 256: kv3_decode_kernel<8><<<g, 256, 0, s>>>(codes, scales, T, x, ldx, cb, r); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qg
