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
//     <= y_j / s, with the thresholds halfway between adjacent levels (an
//     exact tie on the negative side goes to the level of larger magnitude,
//     the mirror image of the positive side);
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
    // the law is symmetric about 0, so are its optimal levels: make it exact
    for (int k = 4; k < 8; ++k) {
        const double m = 0.5 * (lv[k] - lv[7 - k]);
        lv[k] = m;
        lv[7 - k] = -m;
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

// Work split: a vector of D = 32 E values spans E lanes (a "group"; 32 / E
// vectors per warp).  Lane i of a group holds the 16-byte chunks q E + i
// (q = 0..7) of its vector, i.e. local value 4 q + c is element
// j = 4 (q E + i) + c.  Bits 0-1 and the bits above 2 + log2 E of j are thus
// inside a lane (5 butterfly stages in registers) and only the log2 E bits
// of i cross lanes (one shuffle and one fused multiply-add per value and
// stage).  Every warp load or store of a chunk index q touches 32 / E runs of
// 16 E contiguous bytes: whole sectors.
constexpr uint32_t kNibbleLsb = 0x11111111u;

template <int E>
__host__ __device__ constexpr int log2_lanes() { return E == 2 ? 1 : (E == 4 ? 2 : 3); }

// Unnormalised Walsh-Hadamard transform z = H x of the group's vector
// (sg[s] = -1 where lane bit s is set: the upper element of a pair takes p - v).
template <int E>
__device__ __forceinline__ void wht_group(float (&v)[32], const float (&sg)[3]) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1)
#pragma unroll
        for (int a = 0; a < 32; ++a)
            if ((a & h) == 0) {
                const float x0 = v[a], x1 = v[a + h];
                v[a] = x0 + x1;
                v[a + h] = x0 - x1;
            }
#pragma unroll
    for (int st = 0; st < log2_lanes<E>(); ++st)
#pragma unroll
        for (int a = 0; a < 32; ++a) {
            const float p = __shfl_xor_sync(0xffffffffu, v[a], 1 << st);
            v[a] = fmaf(sg[st], v[a], p);
        }
}

template <int E>
__device__ __forceinline__ void group_signs(int lane, float (&sg)[3]) {
#pragma unroll
    for (int st = 0; st < 3; ++st) sg[st] = (st < log2_lanes<E>() && ((lane >> st) & 1)) ? -1.f : 1.f;
}

// The lane's 8 chunks of a vector row (16-byte accesses when vec).
template <int E>
__device__ __forceinline__ void load_chunks(const float* row, int i, bool vec, float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float* p = row + 4 * (q * E + i);
        if (vec) {
            const float4 a = *reinterpret_cast<const float4*>(p);
            v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) v[4 * q + c] = p[c];
        }
    }
}

template <int E>
__device__ __forceinline__ void store_chunks(float* row, int i, bool vec, const float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float* p = row + 4 * (q * E + i);
        if (vec) {
            *reinterpret_cast<float4*>(p) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) p[c] = v[4 * q + c];
        }
    }
}

// Where the lane's local value 4 q + c lands in the bit planes: word
// b E + e, bit L = 4 q + shift, for element j = 4 (q E + i) + c:
//   E = 2: e = c & 1,            L = 4 q + 2 i + (c >> 1)
//   E = 4: e = c,                L = 4 q + i
//   E = 8: e = 4 (i & 1) + c,    L = 4 q + (i >> 1)
template <int E>
__device__ __forceinline__ int plane_shift(int i, int c) {
    if constexpr (E == 2) return 2 * i + (c >> 1);
    else if constexpr (E == 4) return i;
    else return i >> 1;
}

// The words of the three planes a lane reads or writes: 2 per plane at E = 2
// (e = 0, 1), 4 per plane otherwise (e = e0 .. e0 + 3, e0 = 4 (i & 1) at E = 8).
template <int E>
__device__ __forceinline__ int plane_word0(int i) { return E == 8 ? 4 * (i & 1) : 0; }

template <int E>
__device__ __forceinline__ void load_planes(const uint32_t* vec_codes, int i, bool vec, uint32_t (&w)[3][4]) {
    constexpr int NW = E == 2 ? 2 : 4;
#pragma unroll
    for (int b = 0; b < 3; ++b) {
        const uint32_t* p = vec_codes + b * E + plane_word0<E>(i);
        if (vec) {
            if constexpr (NW == 2) {
                const uint2 a = *reinterpret_cast<const uint2*>(p);
                w[b][0] = a.x; w[b][1] = a.y; w[b][2] = 0u; w[b][3] = 0u;
            } else {
                const uint4 a = *reinterpret_cast<const uint4*>(p);
                w[b][0] = a.x; w[b][1] = a.y; w[b][2] = a.z; w[b][3] = a.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) w[b][e] = e < NW ? p[e] : 0u;
        }
    }
}

template <int E>
__device__ __forceinline__ void store_planes(uint32_t* vec_codes, int i, bool vec, const uint32_t (&w)[3][4]) {
    constexpr int NW = E == 2 ? 2 : 4;
#pragma unroll
    for (int b = 0; b < 3; ++b) {
        uint32_t* p = vec_codes + b * E + plane_word0<E>(i);
        if (vec) {
            if constexpr (NW == 2) *reinterpret_cast<uint2*>(p) = make_uint2(w[b][0], w[b][1]);
            else *reinterpret_cast<uint4*>(p) = make_uint4(w[b][0], w[b][1], w[b][2], w[b][3]);
        } else {
#pragma unroll
            for (int e = 0; e < NW; ++e) p[e] = w[b][e];
        }
    }
}

// Grid-stride over batches of 32 / E vectors per warp; the next batch of the
// warp is loaded into registers before the current one is transformed.
// xvec / cvec: rows and code rows aligned for 16-byte (8 at E = 2) accesses.
template <int E>
__global__ void __launch_bounds__(256)
kv3_encode_kernel(const float* __restrict__ x, int64_t T, int64_t ldx, uint32_t* __restrict__ codes,
                  float* __restrict__ scales, KvConsts kc, bool xvec, bool cvec) {
    constexpr int D = 32 * E, VPW = 32 / E;
    const int lane = threadIdx.x & 31, g = lane / E, i = lane % E;
    float sg[3];
    group_signs<E>(lane, sg);
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5) * VPW;
    const int64_t first = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * VPW;
    float nxt[32];
    if (first + g < T) load_chunks<E>(x + (first + g) * ldx, i, xvec, nxt);
    for (int64_t base = first; base < T; base += stride) {     // uniform over the warp
        const int64_t t = base + g;
        const bool active = t < T;
        float v[32];
#pragma unroll
        for (int a = 0; a < 32; ++a) v[a] = active ? nxt[a] : 0.f;
        if (t + stride < T) load_chunks<E>(x + (t + stride) * ldx, i, xvec, nxt);
        wht_group<E>(v, sg);
        float ss = 0.f;
#pragma unroll
        for (int a = 0; a < 32; ++a) ss = fmaf(v[a], v[a], ss);
#pragma unroll
        for (int st = 0; st < log2_lanes<E>(); ++st) ss += __shfl_xor_sync(0xffffffffu, ss, 1 << st);
        const float root = sqrtf(ss);               // same value in every lane of the group
        // codes of the lane's values, nibble q of K[c] = code of value 4 q + c.
        // The thresholds are symmetric (t_{6-m} = -t_m, t_3 = 0): with
        // n = #{m = 4..6 : t_m <= |z|}, code = 4 + n for z >= 0 and 3 - n =
        // (4 + n) ^ 7 for z < 0 -- the number of thresholds <= z, except that
        // an exact tie on the negative side goes to the larger magnitude.
        uint32_t K[4] = {0u, 0u, 0u, 0u};
        if (root > 0.f) {
            const float t4 = root * kc.thr_r[4], t5 = root * kc.thr_r[5], t6 = root * kc.thr_r[6];
            uint32_t N[4] = {0u, 0u, 0u, 0u}, S[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int q = 7; q >= 0; --q)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float z = v[4 * q + c], a = fabsf(z);
                    const bool p1 = a >= t5;               // binary search over t4 < t5 < t6
                    const bool p0 = a >= (p1 ? t6 : t4);
                    N[c] = (N[c] << 4) | ((p1 ? 2u : 0u) + (p0 ? 1u : 0u));
                    S[c] = (S[c] << 4) | (z < 0.f ? 7u : 0u);
                }
#pragma unroll
            for (int c = 0; c < 4; ++c) K[c] = (N[c] | 0x44444444u) ^ S[c];
        }
        // bit planes: this lane's bits, then OR over the lanes sharing a word
        uint32_t w[3][4];
#pragma unroll
        for (int b = 0; b < 3; ++b) {
            if constexpr (E == 2) {
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    w[b][e] = (((K[e] >> b) & kNibbleLsb) << plane_shift<E>(i, e)) |
                              (((K[e + 2] >> b) & kNibbleLsb) << plane_shift<E>(i, e + 2));
                w[b][2] = w[b][3] = 0u;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) w[b][c] = ((K[c] >> b) & kNibbleLsb) << plane_shift<E>(i, c);
            }
        }
#pragma unroll
        for (int st = (E == 8 ? 1 : 0); st < log2_lanes<E>(); ++st)
#pragma unroll
            for (int b = 0; b < 3; ++b)
#pragma unroll
                for (int e = 0; e < (E == 2 ? 2 : 4); ++e) w[b][e] |= __shfl_xor_sync(0xffffffffu, w[b][e], 1 << st);
        if (active) {
            if (i < (E == 8 ? 2 : 1)) store_planes<E>(codes + t * (3 * E), i, cvec, w);
            if (i == 0) scales[t] = root * (1.0f / D);   // exact power-of-two scaling
        }
    }
}

template <int E>
__global__ void __launch_bounds__(256)
kv3_decode_kernel(const uint32_t* __restrict__ codes, const float* __restrict__ scales, int64_t T,
                  float* __restrict__ x, int64_t ldx, KvConsts kc, bool xvec, bool cvec) {
    constexpr int VPW = 32 / E;
    const int lane = threadIdx.x & 31, g = lane / E, i = lane % E;
    float sg[3];
    group_signs<E>(lane, sg);
    float lut = kc.lvl_r[0];                        // lane l (mod 8) holds l_l / sqrt(D)
#pragma unroll
    for (int k = 1; k < 8; ++k) lut = (lane & 7) == k ? kc.lvl_r[k] : lut;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5) * VPW;
    const int64_t first = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * VPW;
    uint32_t nw[3][4];
    float ns = 0.f;
    if (first + g < T) {
        load_planes<E>(codes + (first + g) * (3 * E), i, cvec, nw);
        ns = scales[first + g];
    }
    for (int64_t base = first; base < T; base += stride) {     // uniform over the warp
        const int64_t t = base + g;
        const bool active = t < T;
        uint32_t w[3][4];
#pragma unroll
        for (int b = 0; b < 3; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) w[b][e] = active ? nw[b][e] : 0u;
        const float s = active ? ns : 0.f;
        if (t + stride < T) {
            load_planes<E>(codes + (t + stride) * (3 * E), i, cvec, nw);
            ns = scales[t + stride];
        }
        // nibble q of K[c] = code of the lane's value 4 q + c
        uint32_t K[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int e = E == 2 ? (c & 1) : c;
            const int sh = plane_shift<E>(i, c);
            K[c] = ((w[0][e] >> sh) & kNibbleLsb) | (((w[1][e] >> sh) & kNibbleLsb) << 1) |
                   (((w[2][e] >> sh) & kNibbleLsb) << 2);
        }
        float v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                v[4 * q + c] = s * __shfl_sync(0xffffffffu, lut, (int)((K[c] >> (4 * q)) & 7u));
        wht_group<E>(v, sg);
        if (active) store_chunks<E>(x + t * ldx, i, xvec, v);
    }
}

bool aligned_to(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// 8 warps per block, each taking 32 / E vectors per step.
int grid_vectors(int64_t T, int E) {
    const int64_t per_block = 8 * (32 / E);
    int64_t b = (T + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sm_count() * 8;
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
    const int E = D / 32;
    const int g = grid_vectors(T, E);
    const bool xvec = aligned_to(x, 16) && ldx % 4 == 0;
    const bool cvec = aligned_to(codes, E == 2 ? 8 : 16);
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
    const int E = D / 32;
    const int g = grid_vectors(T, E);
    const bool xvec = aligned_to(x, 16) && ldx % 4 == 0;
    const bool cvec = aligned_to(codes, E == 2 ? 8 : 16);
    switch (D) {
        case 64: kv3_decode_kernel<2><<<g, 256, 0, s>>>(codes, scales, T, x, ldx, kc, xvec, cvec); break;
        case 128: kv3_decode_kernel<4><<<g, 256, 0, s>>>(codes, scales, T, x, ldx, kc, xvec, cvec); break;
        case 256: kv3_decode_kernel<8><<<g, 256, 0, s>>>(codes, scales, T, x, ldx, kc, xvec, cvec); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qg
