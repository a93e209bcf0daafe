// Split-K attention merge ("I wrote a custom CUDA inference engine to run
// Qwen3.5-27B on a $130 mining card", Implementation challenges 3: split-K
// FlashAttention without breaking determinism).  Split s of a row (one head,
// one query) leaves its running max m_s, its sum of exponentials l_s and its
// unnormalised output acc_s [D]; the row's result is
//   m = max_s m_s,  l = sum_s exp(m_s - m) l_s,  o = sum_s exp(m_s - m) acc_s,
//   out = o / l,  lse = m + log(l),
// with binary32 partials, the outputs summed over the splits in index order
// and l in a fixed butterfly, so the result does not depend on how the
// splits were scheduled.  A split that saw
// no key has m_s = -inf and l_s = 0 and contributes nothing; a row whose
// splits are all empty gives out = 0 and lse = -inf.
//
// One warp per row; lanes stride over D with 16-byte loads when D % 4 == 0.
// HBM-bound: S (D + 2) * 4 bytes read and (D + 1) * 4 written per row.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

constexpr int kMaxSplits = 64;

__global__ void __launch_bounds__(256)
splitk_merge_kernel(const float* __restrict__ m, const float* __restrict__ l,
                    const float* __restrict__ acc, int S, int64_t R, int64_t D,
                    float* __restrict__ out, float* __restrict__ lse, bool vec4) {
    __shared__ float wsh[8][kMaxSplits];          // per warp: exp(m_s - m) of its row
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    float* w = wsh[wid];
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + wid; r < R; r += warps) {
        // lanes hold splits lane and lane + 32
        float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
        if (lane < S) { ma = m[(int64_t)lane * R + r]; la = l[(int64_t)lane * R + r]; }
        if (lane + 32 < S) { mb = m[(int64_t)(lane + 32) * R + r]; lb = l[(int64_t)(lane + 32) * R + r]; }
        float mg = fmaxf(ma, mb);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
        const float wa = (ma == -INFINITY) ? 0.f : expf(ma - mg);
        const float wb = (mb == -INFINITY) ? 0.f : expf(mb - mg);
        // l = sum_s w_s l_s: fixed butterfly order (deterministic)
        float lg = fmaf(wb, lb, wa * la);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lg += __shfl_xor_sync(0xffffffffu, lg, o);
        w[lane] = wa;
        w[lane + 32] = wb;
        __syncwarp();
        const bool empty = !(lg > 0.f);
        const float inv = empty ? 0.f : 1.0f / lg;
        if (lane == 0 && lse) lse[r] = empty ? -INFINITY : mg + logf(lg);
        if (vec4) {
            for (int64_t c = lane; c < D / 4; c += 32) {
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int s = 0; s < S; ++s) {
                    const float ws = w[s];
                    const float4 a = *reinterpret_cast<const float4*>(acc + ((int64_t)s * R + r) * D + 4 * c);
                    o.x = fmaf(ws, a.x, o.x);
                    o.y = fmaf(ws, a.y, o.y);
                    o.z = fmaf(ws, a.z, o.z);
                    o.w = fmaf(ws, a.w, o.w);
                }
                *reinterpret_cast<float4*>(out + r * D + 4 * c) =
                    make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
            }
        } else {
            for (int64_t c = lane; c < D; c += 32) {
                float o = 0.f;
                for (int s = 0; s < S; ++s) o = fmaf(w[s], acc[((int64_t)s * R + r) * D + c], o);
                out[r * D + c] = o * inv;
            }
        }
        __syncwarp();                                 // w is rewritten by the next row
    }
}

}  // namespace

int splitk_merge_max_splits() { return kMaxSplits; }

cudaError_t launch_splitk_merge(const float* m, const float* l, const float* acc, int S, int64_t R,
                                int64_t D, float* out, float* lse, cudaStream_t s) {
    const bool vec4 = (D % 4 == 0) && ((uintptr_t)acc % 16 == 0) && ((uintptr_t)out % 16 == 0);
    int64_t grid = (R + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    splitk_merge_kernel<<<(unsigned)grid, 256, 0, s>>>(m, l, acc, S, R, D, out, lse, vec4);
    return cudaGetLastError();
}

}  // namespace qg
