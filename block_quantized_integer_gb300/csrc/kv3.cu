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

// Per-launch constants: the codebook with the 1 / sqrt(D) of the rotation
// folded in, so the kernels run the unnormalised transform z = H x:
//   encode  y = z / sqrt(D), s = sqrt(sum z^2) / D, and y_j / s >= t_k  <=>
//           z_j >= sqrt(sum z^2) * (t_k / sqrt(D))      (s > 0);
//   decode  x^ = H (s * l_k / sqrt(D)).
// Both sides are products of binary32 values rounded once (t_k / sqrt(D) and
// l_k / sqrt(D) are rounded from binary64 on the host).
struct KvConsts {
    float thr_r[7];      // t_k / sqrt(D)
    float lvl_r[8];      // l_k / sqrt(D)
};

KvConsts make_consts(int D) {
    const Codebook& cb = codebook();
    const double r = 1.0 / sqrt((double)D);
    KvConsts c;
    for (int k = 0; k < 7; ++k) c.thr_r[k] = (float)((double)cb.thr[k] * r);
    for (int k = 0; k < 8; ++k) c.lvl_r[k] = (float)((double)cb.level[k] * r);
    return c;
}

// In-warp unnormalised Walsh-Hadamard transform of D = 32 E values, lane L
// holding elements L E .. L E + E - 1: butterflies below E inside the lane,
// the others across lanes, one shuffle and one fused multiply-add each
// (sg[i] = -1 where lane bit i is set: the upper element takes p - v).
template <int E>
__device__ __forceinline__ void wht_warp(float (&v)[E], const float (&sg)[5]) {
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
    for (int i = 0; i < 5; ++i)
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float p = __shfl_xor_sync(0xffffffffu, v[e], 1 << i);
            v[e] = fmaf(sg[i], v[e], p);
        }
}

__device__ __forceinline__ void lane_signs(int lane, float (&sg)[5]) {
#pragma unroll
    for (int i = 0; i < 5; ++i) sg[i] = (lane >> i) & 1 ? -1.f : 1.f;
}

// E consecutive binary32 values of a lane (one 8- or 16-byte access each
// 2 or 4 values when vec, else scalar).
template <int E>
__device__ __forceinline__ void load_lane(const float* p, bool vec, float (&v)[E]) {
    if (vec) {
        if constexpr (E == 2) {
            const float2 a = *reinterpret_cast<const float2*>(p);
            v[0] = a.x; v[1] = a.y;
        } else {
#pragma unroll
            for (int q = 0; q < E / 4; ++q) {
                const float4 a = *reinterpret_cast<const float4*>(p + 4 * q);
                v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = p[e];
    }
}

template <int E>
__device__ __forceinline__ void store_lane(float* p, bool vec, const float (&v)[E]) {
    if (vec) {
        if constexpr (E == 2) {
            *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
        } else {
#pragma unroll
            for (int q = 0; q < E / 4; ++q)
                *reinterpret_cast<float4*>(p + 4 * q) =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) p[e] = v[e];
    }
}

// The 3 E code words of one vector (3 E / 2 8-byte or 3 E / 4 16-byte
// accesses when vec, else scalar).
template <int NW>
__device__ __forceinline__ void load_words(const uint32_t* p, bool vec, uint32_t (&w)[NW]) {
    if (vec) {
        if constexpr (NW % 4 == 0) {
#pragma unroll
            for (int q = 0; q < NW / 4; ++q) {
                const uint4 a = *reinterpret_cast<const uint4*>(p + 4 * q);
                w[4 * q] = a.x; w[4 * q + 1] = a.y; w[4 * q + 2] = a.z; w[4 * q + 3] = a.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < NW / 2; ++q) {
                const uint2 a = *reinterpret_cast<const uint2*>(p + 2 * q);
                w[2 * q] = a.x; w[2 * q + 1] = a.y;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < NW; ++i) w[i] = p[i];
    }
}

template <int NW>
__device__ __forceinline__ void store_words(uint32_t* p, bool vec, const uint32_t (&w)[NW]) {
    if (vec) {
        if constexpr (NW % 4 == 0) {
#pragma unroll
            for (int q = 0; q < NW / 4; ++q)
                *reinterpret_cast<uint4*>(p + 4 * q) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        } else {
#pragma unroll
            for (int q = 0; q < NW / 2; ++q)
                *reinterpret_cast<uint2*>(p + 2 * q) = make_uint2(w[2 * q], w[2 * q + 1]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NW; ++i) p[i] = w[i];
    }
}

// One warp per vector; the next vector of the warp is loaded into registers
// before the current one is transformed.  xvec / cvec: x rows and code rows
// aligned for vector accesses.
template <int E>
__global__ void __launch_bounds__(256)
kv3_encode_kernel(const float* __restrict__ x, int64_t T, int64_t ldx, uint32_t* __restrict__ codes,
                  float* __restrict__ scales, KvConsts kc, bool xvec, bool cvec) {
    constexpr int D = 32 * E;
    const int lane = threadIdx.x & 31;
    float sg[5];
    lane_signs(lane, sg);
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    float nxt[E];
    if (t < T) load_lane<E>(x + t * ldx + lane * E, xvec, nxt);
    for (; t < T; t += warps) {
        float v[E];
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = nxt[e];
        if (t + warps < T) load_lane<E>(x + (t + warps) * ldx + lane * E, xvec, nxt);
        wht_warp<E>(v, sg);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float root = sqrtf(ss);               // same value in every lane
        uint32_t w[3 * E];
        if (root > 0.f) {
            float st[7];
#pragma unroll
            for (int k = 0; k < 7; ++k) st[k] = root * kc.thr_r[k];
            // code = number of st_k <= z_j, by binary search over the sorted
            // thresholds; its three steps give the code's bits 2, 1, 0
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const bool b2 = v[e] >= st[3];
                const bool b1 = v[e] >= (b2 ? st[5] : st[1]);
                const bool b0 = v[e] >= (b2 ? (b1 ? st[6] : st[4]) : (b1 ? st[2] : st[0]));
                w[e] = __ballot_sync(0xffffffffu, b0);
                w[E + e] = __ballot_sync(0xffffffffu, b1);
                w[2 * E + e] = __ballot_sync(0xffffffffu, b2);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 3 * E; ++i) w[i] = 0u;
        }
        if (lane == 0) {
            store_words<3 * E>(codes + t * (3 * E), cvec, w);
            scales[t] = root * (1.0f / D);          // exact power-of-two scaling
        }
    }
}

template <int E>
__global__ void __launch_bounds__(256)
kv3_decode_kernel(const uint32_t* __restrict__ codes, const float* __restrict__ scales, int64_t T,
                  float* __restrict__ x, int64_t ldx, KvConsts kc, bool xvec, bool cvec) {
    const int lane = threadIdx.x & 31;
    float sg[5];
    lane_signs(lane, sg);
    float lut = kc.lvl_r[0];                        // lane i (mod 8) holds l_i / sqrt(D)
#pragma unroll
    for (int i = 1; i < 8; ++i) lut = (lane & 7) == i ? kc.lvl_r[i] : lut;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    uint32_t nw[3 * E];
    float ns = 0.f;
    if (t < T) {
        load_words<3 * E>(codes + t * (3 * E), cvec, nw);   // same address in every lane
        ns = scales[t];
    }
    for (; t < T; t += warps) {
        uint32_t w[3 * E];
#pragma unroll
        for (int i = 0; i < 3 * E; ++i) w[i] = nw[i];
        const float s = ns;
        if (t + warps < T) {
            load_words<3 * E>(codes + (t + warps) * (3 * E), cvec, nw);
            ns = scales[t + warps];
        }
        float v[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const uint32_t k = ((w[e] >> lane) & 1u) | (((w[E + e] >> lane) & 1u) << 1) |
                               (((w[2 * E + e] >> lane) & 1u) << 2);
            v[e] = s * __shfl_sync(0xffffffffu, lut, (int)k);
        }
        wht_warp<E>(v, sg);
        store_lane<E>(x + t * ldx + lane * E, xvec, v);
    }
}

bool aligned_to(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

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
    const KvConsts kc = make_consts(D);
    const int g = grid_vectors(T);
    const int E = D / 32;
    const uintptr_t va = E == 2 ? 8 : 16;
    const bool xvec = aligned_to(x, va) && ldx % (E == 2 ? 2 : 4) == 0;
    const bool cvec = aligned_to(codes, va);
    switch (D) {
        case 64: kv3_encode_kernel<2><<<g, 256, 0, s>>>(x, T, ldx, codes, scales, kc, xvec, cvec); break;
        case 128: kv3_encode_kernel<4><<<g, 256, 0, s>>>(x, T, ldx, codes, scales, kc, xvec, cvec); break;
        case 256: kv3_encode_kernel<8><<<g, 256, 0, s>>>(x, T, ldx, codes, scales, kc, xvec, cvec); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_kv3_decode(const uint32_t* codes, const float* scales, int64_t T, int D,
                              float* x, int64_t ldx, cudaStream_t s) {
    const KvConsts kc = make_consts(D);
    const int g = grid_vectors(T);
    const int E = D / 32;
    const uintptr_t va = E == 2 ? 8 : 16;
    const bool xvec = aligned_to(x, va) && ldx % (E == 2 ? 2 : 4) == 0;
    const bool cvec = aligned_to(codes, va);
    switch (D) {
        case 64: kv3_decode_kernel<2><<<g, 256, 0, s>>>(codes, scales, T, x, ldx, kc, xvec, cvec); break;
        case 128: kv3_decode_kernel<4><<<g, 256, 0, s>>>(codes, scales, T, x, ldx, kc, xvec, cvec); break;
        case 256: kv3_decode_kernel<8><<<g, 256, 0, s>>>(codes, scales, T, x, ldx, kc, xvec, cvec); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qg
