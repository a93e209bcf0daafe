// MoE routing preparation for the grouped GEMM ("A 35B Hybrid-Attention
// Mixture-of-Experts Model on a 6GB 2011 GPU", Methodology 1: the GPU runs a
// grouped 4-bit GEMM for MoE routing during prefill).
//
// From topk_ids [T][topk] (pairs p = token * topk + slot) it builds, in one
// block of 32 warps:
//   counts[e]        pairs routed to expert e,
//   offsets[e]       exclusive prefix sum of counts (offsets[E] = routed pairs),
//   perm[...]        pair indices grouped by expert, (token, slot) order inside
//                    an expert (a stable counting sort),
//   tile_offsets[e]  exclusive prefix sum of ceil(counts[e] / bm) (optional),
//   the m-tile table of the tensor-core grouped GEMM (optional),
// and zeroes the output rows of pairs whose expert id is out of range
// (optional), counting them in *d_err without trapping.
//
// Stability without a global sort: warp w owns the contiguous slice w of the
// pairs (read from a shared-memory copy of the ids when they fit).  Phase 1
// counts experts per warp; phase 2 turns the per-warp counts into starting
// positions (expert-major, then warp order); phase 3 walks each slice in order
// 32 pairs at a time, ranks equal experts inside the step with
// __match_any_sync, and advances the warp's private cursor of each expert.
#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

constexpr int kRouteWarps = 32;
constexpr int kMaxExperts = 1024;
constexpr int64_t kStageBytes = 160 * 1024;   // shared memory the ids may be staged in, with the counts

__device__ __forceinline__ int width_class(int32_t rows) { return rows > 64 ? 0 : (rows > 32 ? 1 : 2); }

// The m-tile table of the tensor-core grouped GEMM, from the exclusive offsets
// off[0..E] (shared memory): per expert its full bm-row tiles and a tail of
// more than 64 rows in class 0, a shorter tail in class 1 (33-64 rows) or 2
// (at most 32), the classes one after another and each in expert order;
// entry {first sorted row, rows, expert, 0}.  Tiles of one width class then
// follow each other in the GEMM's tile order.  The whole block calls it.
__device__ void build_tile_table(const int32_t* __restrict__ off, int32_t E, int bm, int4* __restrict__ table) {
    __shared__ int32_t part[3][32];
    __shared__ int32_t run[3];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    auto counts = [&](int e, int32_t (&c)[3]) {
        c[0] = c[1] = c[2] = 0;
        if (e >= E) return;
        const int32_t n = off[e + 1] - off[e], tail = n % bm;
        c[0] = n / bm;
        if (tail > 0) ++c[width_class(tail)];
    };
    // exclusive block scan of c per class; tot = the chunk's totals
    auto block_scan = [&](int32_t (&c)[3], int32_t (&ex)[3], int32_t (&tot)[3]) {
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            int32_t v = c[k];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (lane == 31) part[k][wid] = v;
            ex[k] = v - c[k];
        }
        __syncthreads();
        if (wid == 0) {
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                int32_t v = lane < nw ? part[k][lane] : 0;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int32_t u = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += u;
                }
                part[k][lane] = v;                      // inclusive over warps
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            ex[k] += wid > 0 ? part[k][wid - 1] : 0;
            tot[k] = part[k][31];
        }
        __syncthreads();                                // part is reused by the next chunk
    };
    int32_t size[3] = {0, 0, 0};                        // pass 1: class sizes
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        int32_t c[3], ex[3], tot[3];
        counts(e0 + tid, c);
        block_scan(c, ex, tot);
#pragma unroll
        for (int k = 0; k < 3; ++k) size[k] += tot[k];
    }
    if (tid == 0) {
        run[0] = 0;
        run[1] = size[0];
        run[2] = size[0] + size[1];
    }
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {          // pass 2: placement
        const int e = e0 + tid;
        int32_t c[3], ex[3], tot[3];
        counts(e, c);
        block_scan(c, ex, tot);
        if (e < E) {
            const int32_t first = off[e], end = off[e + 1];
            int32_t m0 = first;
            int32_t at = run[0] + ex[0];
            for (; end - m0 > 64; m0 += bm) table[at++] = make_int4(m0, min(bm, end - m0), e, 0);
            if (end > m0) {
                const int k = width_class(end - m0);
                table[run[k] + ex[k]] = make_int4(m0, end - m0, e, 0);
            }
        }
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int k = 0; k < 3; ++k) run[k] += tot[k];
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kRouteWarps * 32)
moe_route_kernel(const int32_t* __restrict__ ids, int64_t P, int32_t E,
                 int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ perm, int32_t* __restrict__ tile_offsets, int bm,
                 int4* __restrict__ table, float* __restrict__ y, int64_t N,
                 int32_t* __restrict__ d_err, bool staged) {
    extern __shared__ int32_t cnt[];          // [kRouteWarps][E], scans [E+1] x 2, staged ids [P]
    int32_t* scan = cnt + kRouteWarps * E;
    int32_t* tscan = scan + (E + 1);
    int32_t* sid = tscan + (E + 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t L = (P + kRouteWarps - 1) / kRouteWarps;
    const int64_t s0 = min64(P, warp * L), s1 = min64(P, s0 + L);
    pdl_wait();                               // the ids may come from the previous kernel
    pdl_release();

    // When they fit, the ids are first copied into shared memory by the whole
    // block, four loads in flight a thread: both walks over a warp's slice then
    // read shared memory instead of waiting on one global load per step.
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
    if (table != nullptr) build_tile_table(scan, E, bm, table);
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
                             int32_t* tile_offsets, int bm, int4* tile_table, float* y, int64_t N,
                             int32_t* d_err, cudaStream_t s) {
    if (E > kMaxExperts) return cudaErrorInvalidValue;
    const int64_t P = T * topk;
    const int64_t base = (kRouteWarps * (int64_t)E + 2 * (E + 1)) * 4;
    const bool staged = base + P * 4 <= kStageBytes;
    const int smem = (int)(base + (staged ? P * 4 : 0));
    cudaError_t e = ensure_smem_attr((const void*)moe_route_kernel, smem, 8);
    if (e != cudaSuccess) return e;
    return launch_pdl(moe_route_kernel, dim3(1), dim3(kRouteWarps * 32), (size_t)smem, s, topk_ids, P,
                      E, counts, offsets, perm, tile_offsets, bm < 1 ? 1 : bm, tile_table, y, N, d_err,
                      staged);
}

}  // namespace qg
