// Tile GEMM on warp-level int8 MMA (mma.sync m16n8k32 s8.s8 -> s32).
//
// One m16n8k32 instruction spans exactly one 32-element quantization group,
// so each accumulator it produces is the exact group dot product S of a 16x8
// block of outputs; the warp scales it by dx[m,g] * dw[n,g] into binary32
// accumulators at once.  This is the int8 tile path of the mining-card engine
// ("I wrote a custom CUDA inference engine to run Qwen3.5-27B on a $130 mining
// card", Features: hand-written Q8_0 GEMM tiles on int8 dot products) moved
// from dp4a onto warp MMA.  On sm_103a it is the legacy tensor path: the
// baseline the tcgen05 kernel is measured against, the kernel for mid-sized
// M, and the grouped MoE GEMM ("A 35B Hybrid-Attention Mixture-of-Experts
// Model on a 6GB 2011 GPU", Methodology 1: grouped 4-bit GEMM for MoE
// routing) whose A rows are gathered through the routing permutation.
//
// CTA tile 128 x 128; K staged 64 bytes (two groups) at a time through a
// 4-deep cp.async ring (zero-filled past the edges); scales of a stage are
// loaded into registers one iteration ahead and parked in shared memory as
// binary32.  8 warps in a 2 x 4 grid, 64 x 32 outputs per warp.
#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4, THREADS = 256;
constexpr int A_BYTES = BM * BK;            // int8 activations
constexpr int DX_BYTES = BM * 2 * 4;        // two groups of binary32 scales
constexpr int DW_BYTES = BN * 2 * 4;        // two groups, stored as binary32

template <bool kQ4>
struct Smem {
    static constexpr int kB = kQ4 ? BN * BK / 2 : BN * BK;
    static constexpr int kStage = A_BYTES + kB + DX_BYTES + DW_BYTES;
    static constexpr int kTotal = kStage * STAGES + BM * 4;   // + tile row map
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte cp.async with zero fill (src-size 0 writes zeros, reads nothing).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
    const int n = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void mma_s8(int (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0), "r"(0),
          "r"(0), "r"(0));
}

// 16-byte chunk c (0..3) of row r in a 64-byte-row tile, swizzled so that the
// 8 rows x 16 bytes of one ldmatrix land in 8 different bank groups.
__device__ __forceinline__ int sw64(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }
// 16-byte half h (0..1) of row r in a 32-byte-row tile (packed 4-bit rows).
__device__ __forceinline__ int sw32(int r, int h) { return r * 32 + ((h ^ ((r >> 2) & 1)) << 4); }

template <bool kQ4, bool kGather>
__global__ void __launch_bounds__(THREADS, 1)
mma_gemm_kernel(const int8_t* __restrict__ qx, const float* __restrict__ dx, int64_t M,
                int64_t N, int64_t K, const uint8_t* __restrict__ qw,
                const uint16_t* __restrict__ dw, float* __restrict__ y, int64_t ldy,
                GatherArgs ga, int n_tiles, bool vec2) {
    extern __shared__ __align__(128) uint8_t smem[];
    using S = Smem<kQ4>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int warp_m = warp >> 2, warp_n = warp & 3;
    const int64_t G = K / kGroup;
    int32_t* rowmap = reinterpret_cast<int32_t*>(smem + S::kStage * STAGES);

    // ---- which tile -----------------------------------------------------------
    int64_t m0 = 0, rows = 0, n0 = 0;
    const uint8_t* wbase = qw;
    const uint16_t* dwbase = dw;
    if constexpr (kGather) {
        const int64_t t = blockIdx.x;
        const int64_t mt_glob = t / n_tiles;
        n0 = (t % n_tiles) * BN;
        if (mt_glob >= ga.tile_offsets[ga.E]) return;   // uniform over the block
        int lo = 0, hi = ga.E - 1;                       // last e: tile_offsets[e] <= mt
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ga.tile_offsets[mid] <= mt_glob) lo = mid; else hi = mid - 1;
        }
        const int e = lo;
        const int64_t seg = ga.offsets[e] + (mt_glob - ga.tile_offsets[e]) * BM;
        rows = min64(BM, (int64_t)ga.offsets[e + 1] - seg);
        wbase = qw + (int64_t)e * N * (kQ4 ? K / 2 : K);
        dwbase = dw + (int64_t)e * N * G;
        if (tid < BM) rowmap[tid] = tid < rows ? ga.perm[seg + tid] : -1;
    } else {
        m0 = (int64_t)blockIdx.y * BM;
        n0 = (int64_t)blockIdx.x * BN;
        rows = min64(BM, M - m0);
        if (tid < BM) rowmap[tid] = tid < rows ? (int32_t)tid : -1;
    }
    __syncthreads();

    // activation row of tile row r (or -1 past the tile's rows)
    auto xrow = [&](int r) -> int64_t {
        const int32_t v = rowmap[r];
        if (v < 0) return -1;
        if constexpr (kGather) return ga.x_row_mode ? (int64_t)v : (int64_t)(v / ga.topk);
        else return m0 + v;
    };

    const int64_t kstages = (K + BK - 1) / BK;
    const uint32_t sbase = smem_u32(smem);

    auto load_tiles = [&](int64_t ks, int slot) {
        const uint32_t st = sbase + slot * S::kStage;
        const int64_t kb = ks * BK;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int idx = tid + i * THREADS;
            const int r = idx >> 2, c = idx & 3;
            const int64_t xr = xrow(r);
            const bool ok = xr >= 0 && kb + c * 16 < K;
            cp_async16(st + sw64(r, c), ok ? (const void*)(qx + xr * K + kb + c * 16) : qx, ok);
        }
        const uint32_t sb = st + A_BYTES;
        if constexpr (!kQ4) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int idx = tid + i * THREADS;
                const int r = idx >> 2, c = idx & 3;
                const bool ok = n0 + r < N && kb + c * 16 < K;
                cp_async16(sb + sw64(r, c),
                           ok ? (const void*)(wbase + (n0 + r) * K + kb + c * 16) : wbase, ok);
            }
        } else {
            const int r = tid >> 1, h = tid & 1;
            const bool ok = n0 + r < N && kb + h * 32 < K;
            cp_async16(sb + sw32(r, h),
                       ok ? (const void*)(wbase + (n0 + r) * (K / 2) + kb / 2 + h * 16) : wbase,
                       ok);
        }
    };
    // two binary32 scales of one stage for this thread's row (t < 128: dx of
    // tile row t; t >= 128: dw of tile column t - 128)
    auto fetch_scales = [&](int64_t ks) -> float2 {
        const int64_t g0 = ks * BK / kGroup;
        float2 v = make_float2(0.f, 0.f);
        if (tid < BM) {
            const int64_t xr = xrow(tid);
            if (xr >= 0) {
                v.x = dx[xr * G + g0];
                if (g0 + 1 < G) v.y = dx[xr * G + g0 + 1];
            }
        } else {
            const int64_t n = n0 + tid - BM;
            if (n < N) {
                v.x = half_bits_to_float(dwbase[n * G + g0]);
                if (g0 + 1 < G) v.y = half_bits_to_float(dwbase[n * G + g0 + 1]);
            }
        }
        return v;
    };
    auto park_scales = [&](int slot, float2 v) {
        float* p = reinterpret_cast<float*>(smem + slot * S::kStage + A_BYTES + S::kB);
        // dx region [BM][2] followed by the dw region [BN][2]
        reinterpret_cast<float2*>(p)[tid] = v;
    };

    float acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[i][j][k] = 0.f;

    // ---- prologue -------------------------------------------------------------
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < kstages) {
            load_tiles(s, s);
            park_scales(s, fetch_scales(s));
        }
        cp_commit();
    }

    // ---- main loop ------------------------------------------------------------
    for (int64_t ks = 0; ks < kstages; ++ks) {
        cp_wait<STAGES - 2>();
        __syncthreads();
        const int64_t nk = ks + STAGES - 1;
        float2 pending = make_float2(0.f, 0.f);
        if (nk < kstages) {
            load_tiles(nk, (int)(nk % STAGES));
            pending = fetch_scales(nk);
        }
        cp_commit();

        const int slot = (int)(ks % STAGES);
        const uint32_t sa = sbase + slot * S::kStage;
        const uint32_t sb = sa + A_BYTES;
        const float* sdx = reinterpret_cast<const float*>(smem + slot * S::kStage + A_BYTES + S::kB);
        const float* sdw = sdx + BM * 2;
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
            uint32_t a[4][4];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int r = warp_m * 64 + mt * 16 + (lane & 15);
                ldsm_x4(sa + sw64(r, 2 * gi + (lane >> 4)), a[mt][0], a[mt][1], a[mt][2], a[mt][3]);
            }
            uint32_t b[4][2];
            if constexpr (!kQ4) {
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    const int r = warp_n * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    ldsm_x4(sb + sw64(r, 2 * gi + ((lane >> 3) & 1)), b[2 * np][0], b[2 * np][1],
                            b[2 * np + 1][0], b[2 * np + 1][1]);
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int r = warp_n * 32 + nt * 8 + (lane >> 2);
                    const uint32_t wv = lds32(sb + sw32(r, gi) + (lane & 3) * 4);
                    b[nt][0] = nib_to_s8(wv & 0x0f0f0f0fu);          // elements k .. k+3
                    b[nt][1] = nib_to_s8((wv >> 4) & 0x0f0f0f0fu);   // elements k+16 ..
                }
            }
            float sx[4][2], sw[4][2];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int r = warp_m * 64 + mt * 16 + (lane >> 2);
                sx[mt][0] = sdx[r * 2 + gi];
                sx[mt][1] = sdx[(r + 8) * 2 + gi];
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int c = warp_n * 32 + nt * 8 + (lane & 3) * 2;
                sw[nt][0] = sdw[c * 2 + gi];
                sw[nt][1] = sdw[(c + 1) * 2 + gi];
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    int c[4];
                    mma_s8(c, a[mt], b[nt][0], b[nt][1]);
                    acc[mt][nt][0] = fmaf(__int2float_rn(c[0]), sx[mt][0] * sw[nt][0], acc[mt][nt][0]);
                    acc[mt][nt][1] = fmaf(__int2float_rn(c[1]), sx[mt][0] * sw[nt][1], acc[mt][nt][1]);
                    acc[mt][nt][2] = fmaf(__int2float_rn(c[2]), sx[mt][1] * sw[nt][0], acc[mt][nt][2]);
                    acc[mt][nt][3] = fmaf(__int2float_rn(c[3]), sx[mt][1] * sw[nt][1], acc[mt][nt][3]);
                }
        }
        if (nk < kstages) park_scales((int)(nk % STAGES), pending);
    }
    cp_wait<0>();

    // ---- epilogue -------------------------------------------------------------
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = warp_m * 64 + mt * 16 + (lane >> 2) + h * 8;
            const int32_t v = rowmap[r];
            if (v < 0) continue;
            const int64_t orow = kGather ? (int64_t)v : m0 + v;
            float* yr = y + orow * ldy;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int64_t c = n0 + warp_n * 32 + nt * 8 + (lane & 3) * 2;
                const float v0 = acc[mt][nt][2 * h], v1 = acc[mt][nt][2 * h + 1];
                if (vec2 && c + 1 < N) {
                    *reinterpret_cast<float2*>(yr + c) = make_float2(v0, v1);
                } else if (c + 1 < N) {
                    yr[c] = v0;
                    yr[c + 1] = v1;
                } else if (c < N) {
                    yr[c] = v0;
                }
            }
        }
}

template <bool kQ4, bool kGather>
cudaError_t launch(dim3 grid, const int8_t* qx, const float* dx, int64_t M, int64_t N,
                   int64_t K, const uint8_t* qw, const uint16_t* dw, float* y, int64_t ldy,
                   GatherArgs ga, int n_tiles, cudaStream_t s) {
    constexpr int smem = Smem<kQ4>::kTotal;
    cudaError_t e = ensure_smem_attr((const void*)mma_gemm_kernel<kQ4, kGather>, smem,
                                     (kQ4 ? 1 : 0) + (kGather ? 2 : 0));
    if (e != cudaSuccess) return e;
    const bool vec2 = ((uintptr_t)y % 8 == 0) && (ldy % 2 == 0);
    mma_gemm_kernel<kQ4, kGather><<<grid, THREADS, smem, s>>>(qx, dx, M, N, K, qw, dw, y, ldy,
                                                               ga, n_tiles, vec2);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mma_gemm(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                            const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                            cudaStream_t s) {
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    GatherArgs ga{};
    const uint8_t* w = (const uint8_t*)qw;
    return q4 ? launch<true, false>(grid, qx, dx, M, N, K, w, dw, y, ldy, ga, 0, s)
              : launch<false, false>(grid, qx, dx, M, N, K, w, dw, y, ldy, ga, 0, s);
}

int mma_tile_m() { return BM; }

cudaError_t launch_mma_grouped(const int8_t* qx, const float* dx, int64_t P, int64_t N,
                               int64_t K, const uint8_t* qw4, const uint16_t* dw, float* y,
                               const GatherArgs& ga, cudaStream_t s) {
    const int n_tiles = (int)((N + BN - 1) / BN);
    // upper bound on m-tiles: sum_e ceil(c_e / BM) <= P / BM + E
    const int64_t mt_max = P / BM + ga.E;
    dim3 grid((unsigned)(mt_max * n_tiles));
    return launch<true, true>(grid, qx, dx, 0, N, K, qw4, dw, y, N, ga, n_tiles, s);
}

}  // namespace qg
