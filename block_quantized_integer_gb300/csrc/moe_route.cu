// MoE routing preparation for the grouped GEMM ("A 35B Hybrid-Attention
// Mixture-of-Experts Model on a 6GB 2011 GPU", Methodology 1: the GPU runs a
// grouped 4-bit GEMM for MoE routing during prefill).
//
// From topk_ids [T][topk] (pairs p = token * topk + slot) it builds, in one
// block of 16 warps:
//   counts[e]        pairs routed to expert e,
//   offsets[e]       exclusive prefix sum of counts (offsets[E] = routed pairs),
//   perm[...]        pair indices grouped by expert, (token, slot) order inside
//                    an expert (a stable counting sort),
//   tile_offsets[e]  exclusive prefix sum of ceil(counts[e] / bm) (optional),
// and zeroes the output rows of pairs whose expert id is out of range
// (optional), counting them in *d_err without trapping.
//
// Stability without a global sort: warp w owns the contiguous slice w of the
// pairs (read from a shared-memory copy of the ids when they fit).  Phase 1 counts experts per warp; phase 2 turns the per-warp counts
// into starting positions (expert-major, then warp order); phase 3 walks each
// slice in order 32 pairs at a time, ranks equal experts inside the step with
// __match_any_sync, and advances the warp's private cursor of each expert.
#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

constexpr int kRouteWarps = 16;
constexpr int kMaxExperts = 1024;
constexpr int64_t kStageMax = 32768;      // routed pairs whose ids are staged in shared memory

__global__ void __launch_bounds__(kRouteWarps * 32)
moe_route_kernel(const int32_t* __restrict__ ids, int64_t P, int32_t E,
                 int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ perm, int32_t* __restrict__ tile_offsets, int bm,
                 float* __restrict__ y, int64_t N, int32_t* __restrict__ d_err) {
    extern __shared__ int32_t cnt[];          // [kRouteWarps][E], scans [E+1] x 2, staged ids [P]
    int32_t* scan = cnt + kRouteWarps * E;
    int32_t* tscan = scan + (E + 1);
    int32_t* sid = tscan + (E + 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t L = (P + kRouteWarps - 1) / kRouteWarps;
    const int64_t s0 = min64(P, warp * L), s1 = min64(P, s0 + L);
    pdl_wait();                               // the ids may come from the previous kernel
    pdl_release();

    // Up to kStageMax pairs, the ids are first copied into shared memory by
    // the whole block, four loads in flight a thread: both walks over a warp's
    // slice then read shared memory instead of waiting on one global load per
    // step.
    const bool staged = P <= kStageMax;
    if (staged) {
        for (int64_t i0 = tid; i0 < P; i0 += 4 * (int64_t)blockDim.x) {
            int32_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t i = i0 + u * (int64_t)blockDim.x;
                v[u] = i < P ? ids[i] : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t i = i0 + u * (int64_t)blockDim.x;
                if (i < P) sid[i] = v[u];
            }
        }
    }
    const int32_t* src = staged ? sid : ids;
    for (int i = tid; i < kRouteWarps * E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();

    // phase 1: per-warp expert counts; unrouted pairs counted into d_err
    int bad = 0;
    for (int64_t p = s0 + lane; p < s1; p += 32) {
        const int32_t e = src[p];
        if (e >= 0 && e < E) atomicAdd(&cnt[warp * E + e], 1);
        else ++bad;
    }
    if (bad) atomicAdd(d_err, bad);
    __syncthreads();

    // phase 2: totals, exclusive scans over experts, per-warp start positions
    for (int e = tid; e < E; e += blockDim.x) {
        int32_t t = 0;
        for (int w = 0; w < kRouteWarps; ++w) t += cnt[w * E + e];
        scan[e] = t;
        tscan[e] = (t + bm - 1) / bm;
    }
    __syncthreads();
    if (warp == 0) {
        // sequential-in-chunks scan by one warp: 32 experts per step
        int32_t run = 0, trun = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            int32_t v = e < E ? scan[e] : 0, tv = e < E ? tscan[e] : 0;
            int32_t incl = v, tincl = tv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t a = __shfl_up_sync(0xffffffffu, incl, o);
                const int32_t b = __shfl_up_sync(0xffffffffu, tincl, o);
                if (lane >= o) { incl += a; tincl += b; }
            }
            if (e < E) {
                counts[e] = v;
                scan[e] = run + incl - v;      // exclusive
                tscan[e] = trun + tincl - tv;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
            trun += __shfl_sync(0xffffffffu, tincl, 31);
        }
        if (lane == 0) { scan[E] = run; tscan[E] = trun; }
    }
    __syncthreads();
    for (int e = tid; e <= E; e += blockDim.x) {
        offsets[e] = scan[e];
        if (tile_offsets) tile_offsets[e] = tscan[e];
    }
    // cnt[w][e] becomes warp w's first position for expert e
    for (int e = tid; e < E; e += blockDim.x) {
        int32_t pos = scan[e];
        for (int w = 0; w < kRouteWarps; ++w) {
            const int32_t c = cnt[w * E + e];
            cnt[w * E + e] = pos;
            pos += c;
        }
    }
    __syncthreads();

    // phase 3: stable placement, 32 pairs per step in slice order
    const unsigned lt = (1u << lane) - 1u;
    for (int64_t base = s0; base < s1; base += 32) {
        const int64_t p = base + lane;
        int32_t e = p < s1 ? src[p] : -1;
        const bool ok = e >= 0 && e < E;
        if (!ok) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (ok) {
            const int32_t pos = cnt[warp * E + e] + __popc(peers & lt);
            perm[pos] = (int32_t)p;
        }
        __syncwarp();
        if (ok && (peers & lt) == 0) cnt[warp * E + e] += __popc(peers);
        __syncwarp();
        if (!ok && p < s1 && y != nullptr) {
            for (int64_t n = 0; n < N; ++n) y[p * N + n] = 0.f;
        }
    }
}

}  // namespace

cudaError_t launch_moe_route(const int32_t* topk_ids, int64_t T, int32_t topk, int32_t E,
                             int32_t* counts, int32_t* offsets, int32_t* perm,
                             int32_t* tile_offsets, int bm, float* y, int64_t N,
                             int32_t* d_err, cudaStream_t s) {
    if (E > kMaxExperts) return cudaErrorInvalidValue;
    const int64_t P = T * topk;
    const int smem = (int)((kRouteWarps * E + 2 * (E + 1) + (P <= kStageMax ? P : 0)) * 4);
    cudaError_t e = ensure_smem_attr((const void*)moe_route_kernel, smem, 8);
    if (e != cudaSuccess) return e;
    return launch_pdl(moe_route_kernel, dim3(1), dim3(kRouteWarps * 32), (size_t)smem, s, topk_ids, P,
                      E, counts, offsets, perm, tile_offsets, bm < 1 ? 1 : bm, y, N, d_err);
}

}  // namespace qg
