// Prefill GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// y[m,n] = sum_g dw[n,g] dx[m,g] S[m,n,g] with S the exact integer dot
// product of one 32-group ("I wrote a custom CUDA inference engine to run
// Qwen3.5-27B on a $130 mining card", Features: the Q8_0 GEMM tile path of the
// prefill; "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU",
// Methodology 1: grouped 4-bit GEMM for MoE routing; Methodology 4: one pass
// over the whole prompt keeps the GEMM M large).
//
// sm_103a has no integer tcgen05 MMA form, so the codes are widened to
// binary16, where every value in [-127, 127] is exact, and multiplied with
// kind::f16 into binary32 tensor memory: each product is an integer below
// 2^14 and each group sum an integer below 2^19, which the tensor core
// accumulates without loss (the group-dot tests check this bit for bit).
//
// Per CTA: a 128 x 128 output tile, K walked one 32-group at a time.
//   pre-pass    activation codes widened to binary16 once per call (for the
//               MoE product also gathered into expert order with their scales).
//   warp 8      TMA producer: binary16 A tiles (2 groups per stage, 128-byte
//               swizzle, the operand layout the MMA reads directly), int8 or
//               packed 4-bit B tiles (4 / 8 groups per stage, 128-byte
//               swizzle), dx / dw scale tiles every 8 groups.
//   warps 10-11 converters: B codes -> binary16 into the canonical K-major
//               no-swizzle layout (8 x 16-byte core matrices), one group per
//               buffer, 4 buffers; dw -> binary32 once per 8 groups.
//   warp 9      one thread issues two K=16 MMAs per group into one of four
//               128-column TMEM buffers (the first MMA overwrites).
//   warps 0-7   epilogue: one tcgen05.ld round trip fetches a group's 64
//               partials per thread (row = TMEM lane, warpgroup = 64 columns);
//               the buffer is released at once and y += S * (dx * dw) runs on
//               packed f32x2 instructions into binary32 registers.
// Every mbarrier wait is bounded; on a timeout the CTA sets a device error
// word, drains its own TMA copies and MMAs, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace qg {

__device__ unsigned int g_tc_error = 0;

namespace {

using namespace tc;

constexpr int BM = 128, BN = 128;
constexpr int GA = 2;                  // groups per A stage = one pair (64 binary16 = 128-byte rows)
constexpr int NO = 4;                  // operand slots: binary16 A stage + binary16 B pair
constexpr int NB = 4;                  // B code stages (each 128-byte rows: 4 Q8 / 8 Q4 groups)
constexpr int NP = 2;                  // TMEM pair slots (two 128-column accumulators each)
constexpr int SCG = 8;                 // groups per scale stage
constexpr int NSC = 3;                 // scale stages
constexpr int EPI_WARPS = 16;          // 4 per TMEM lane quarter, 32 columns each
constexpr int PROD_WARP = 16, MMA_WARP = 17, CONV_WARP0 = 18, CONV_WARPS = 2;
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int THREADS = (CONV_WARP0 + CONV_WARPS) * 32;   // 640

constexpr int A_STAGE = BM * 128;                    // 16384
constexpr int B_STAGE = BN * 128;                    // 16384
constexpr int F16_B = BN * 32 * 2;                   // 8192: one group of binary16 B
constexpr int F16_PAIR = 2 * F16_B;                  // 16384
constexpr int SC_DX = BM * SCG * 4;                  // 4096: dx [8][128] f32 (dense) or [128][8] (grouped)
constexpr int SC_DW = SCG * BN * 4;                  // 4096: dw [8][128] f32 (transposed)
constexpr int SC_STAGE = SC_DX + SC_DW;              // 8192

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + NO * A_STAGE;
constexpr int OFF_F16 = OFF_B + NB * B_STAGE;
constexpr int OFF_SC = OFF_F16 + NO * F16_PAIR;
constexpr int OFF_BAR = OFF_SC + NSC * SC_STAGE;
constexpr int NUM_BARS = 3 * NO + 2 * NB + 2 * NP + 2 * NSC + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;     // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_B % 1024 == 0 && OFF_F16 % 1024 == 0, "swizzled stages need 1 KiB alignment");

constexpr uint32_t TMEM_COLS = NP * 2 * BN;          // 512: two pair slots of two groups
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
constexpr uint32_t kSpinLimit = 1u << 22;          // drain polls after an abort
constexpr long long kWaitCycles = 4000000000ll;      // ~2 s at 2 GHz: a wait that long has failed
constexpr uint32_t kSleepHintNs = 20000;             // a waiter sleeps until the phase flips

// full_a: TMA A stage landed; full_f16: converters wrote the B pair; ops_free:
// the MMAs that read an operand slot completed (one commit frees A and B).
struct Bars {
    uint32_t full_a, full_f16, ops_free, full_b, empty_b, tfull, tempty, full_sc, empty_sc, drain;
};

__device__ __forceinline__ Bars bars_at(uint32_t base) {
    Bars b;
    b.full_a = base;
    b.full_f16 = b.full_a + 8 * NO;
    b.ops_free = b.full_f16 + 8 * NO;
    b.full_b = b.ops_free + 8 * NO;
    b.empty_b = b.full_b + 8 * NB;
    b.tfull = b.empty_b + 8 * NB;
    b.tempty = b.tfull + 8 * NP;
    b.full_sc = b.tempty + 8 * NP;
    b.empty_sc = b.full_sc + 8 * NSC;
    b.drain = b.empty_sc + 8 * NSC;
    return b;
}

// Bounded wait: the thread sleeps in try_wait until the phase completes; after
// kWaitCycles without completion (or when another role gave up) it returns
// false.  kWarp: all 32 lanes call it and leave together.
template <bool kWarp>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort) {
    bool ok = mbar_try_wait(bar, parity);
    if (kWarp) ok = __all_sync(0xffffffffu, ok);
    if (ok) return true;
    const long long start = clock64();
    for (;;) {
        ok = mbar_try_wait_sleep(bar, parity, kSleepHintNs);
        if (kWarp) ok = __all_sync(0xffffffffu, ok);
        if (ok) return true;
        bool ab = *abort != 0;
        if (kWarp) ab = __any_sync(0xffffffffu, ab);
        if (ab) return false;
        bool late = clock64() - start > kWaitCycles;
        if (kWarp) late = __any_sync(0xffffffffu, late);
        if (late) {
            *abort = 1;
            atomicOr(&g_tc_error, 1u);
            return false;
        }
    }
}

// Bounded wait used only while draining after an abort.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < kSpinLimit; ++it)
        if (mbar_try_wait(bar, parity)) return;
}

// int8 pairs -> binary16 pairs, exactly: (b ^ 0x80) = b + 128 in [1, 255];
// under the exponent byte 0x64 it reads as 1024 + b + 128; minus 1152 gives b.
__device__ __forceinline__ uint32_t s8x2_to_h2(uint32_t t, uint32_t sel) {
    const uint32_t h = __byte_perm(t, 0x64646464u, sel);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}
__device__ __forceinline__ void s8x16_to_h16(const uint4 v, uint4& lo, uint4& hi) {
    const uint32_t a = v.x ^ 0x80808080u, b = v.y ^ 0x80808080u;
    const uint32_t c = v.z ^ 0x80808080u, d = v.w ^ 0x80808080u;
    lo = make_uint4(s8x2_to_h2(a, 0x4140), s8x2_to_h2(a, 0x4342),
                    s8x2_to_h2(b, 0x4140), s8x2_to_h2(b, 0x4342));
    hi = make_uint4(s8x2_to_h2(c, 0x4140), s8x2_to_h2(c, 0x4342),
                    s8x2_to_h2(d, 0x4140), s8x2_to_h2(d, 0x4342));
}
// Q4 nibble pairs (stored q + 8 in [0, 15]) -> binary16 pairs: under 0x64 the
// nibble reads 1024 + s; minus 1032 gives s - 8 = q.
__device__ __forceinline__ uint32_t u4x2_to_h2(uint32_t nib_bytes, uint32_t sel) {
    const uint32_t h = __byte_perm(nib_bytes, 0x64646464u, sel);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64086408u));
    return r;
}

// Group gi (0 .. GB-1) of the int8 / packed 4-bit B stage -> binary16 B buffer
// (canonical no-swizzle K-major layout: core matrix (row/8, k8) at
// (row/8)*512 + k8*128, row%8 at +16 each).
template <bool kQ4>
__device__ __forceinline__ void convert_group(const uint8_t* src, uint8_t* dst, int gi, int ct) {
    if constexpr (!kQ4) {
#pragma unroll 2
        for (int j = 0; j < BN * 2 / CONV_THREADS; ++j) {
            const int i = ct + j * CONV_THREADS;
            const int row = i & (BN - 1), half = i >> 7;
            const int chunk = gi * 2 + half;          // 128-byte swizzle: chunk ^ (row & 7)
            const uint4 v = *reinterpret_cast<const uint4*>(src + row * 128 + ((chunk ^ (row & 7)) << 4));
            uint4 lo, hi;
            s8x16_to_h16(v, lo, hi);
            uint8_t* o = dst + (row >> 3) * 512 + (half * 2) * 128 + (row & 7) * 16;
            *reinterpret_cast<uint4*>(o) = lo;
            *reinterpret_cast<uint4*>(o + 128) = hi;
        }
    } else {
#pragma unroll
      for (int j = 0; j < BN / CONV_THREADS; ++j) {
        const int row = ct + j * CONV_THREADS;        // one 16-byte group per row
        const uint4 v = *reinterpret_cast<const uint4*>(src + row * 128 + ((gi ^ (row & 7)) << 4));
        // byte j: element j (low nibble), element j+16 (high nibble)
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t lo_h[8], hi_h[8];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t l = w[t] & 0x0f0f0f0fu, h = (w[t] >> 4) & 0x0f0f0f0fu;
            lo_h[2 * t] = u4x2_to_h2(l, 0x4140);
            lo_h[2 * t + 1] = u4x2_to_h2(l, 0x4342);
            hi_h[2 * t] = u4x2_to_h2(h, 0x4140);
            hi_h[2 * t + 1] = u4x2_to_h2(h, 0x4342);
        }
        uint8_t* o = dst + (row >> 3) * 512 + (row & 7) * 16;
        *reinterpret_cast<uint4*>(o) = make_uint4(lo_h[0], lo_h[1], lo_h[2], lo_h[3]);
        *reinterpret_cast<uint4*>(o + 128) = make_uint4(lo_h[4], lo_h[5], lo_h[6], lo_h[7]);
        *reinterpret_cast<uint4*>(o + 256) = make_uint4(hi_h[0], hi_h[1], hi_h[2], hi_h[3]);
        *reinterpret_cast<uint4*>(o + 384) = make_uint4(hi_h[4], hi_h[5], hi_h[6], hi_h[7]);
      }
    }
}

struct GroupedArgs {
    const int32_t* perm;          // sorted position -> pair index
    const int32_t* offsets;       // [E+1]
    const int32_t* tile_offsets;  // [E+1] in 128-row tiles
    int32_t E;
    int64_t N;                    // per-expert output columns
};

struct Tile {
    int64_t m0, rows, n0, bn0;    // first A row, valid rows, first column, first B row
    int64_t sg0;                  // first row of the transposed scale plane (expert * G)
};

template <bool kGrouped>
__device__ __forceinline__ Tile tile_at(int64_t t, int64_t M, int G, const GroupedArgs& ga,
                                        int n_tiles) {
    Tile T;
    const int64_t mt = t / n_tiles;
    T.n0 = (t % n_tiles) * BN;
    if constexpr (kGrouped) {
        int lo = 0, hi = ga.E - 1;                       // last e with tile_offsets[e] <= mt
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ga.tile_offsets[mid] <= mt) lo = mid; else hi = mid - 1;
        }
        T.m0 = ga.offsets[lo] + (mt - ga.tile_offsets[lo]) * BM;
        T.rows = min64(BM, (int64_t)ga.offsets[lo + 1] - T.m0);
        T.bn0 = (int64_t)lo * ga.N + T.n0;
        T.sg0 = (int64_t)lo * G;
    } else {
        T.m0 = mt * BM;
        T.rows = min64(BM, M - T.m0);
        T.bn0 = T.n0;
        T.sg0 = 0;
    }
    return T;
}

// Persistent: CTA b takes tiles b, b + gridDim.x, ...  All roles walk the same
// tile sequence; ring positions and barrier phases run on across tiles.
template <bool kQ4, bool kGrouped>
__global__ void __launch_bounds__(THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_dx, const __grid_constant__ CUtensorMap map_dw,
               float* __restrict__ y, int64_t M, int64_t N, int64_t K, int64_t ldy, bool vec4,
               GroupedArgs ga, int n_tiles, int64_t dense_tiles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Bars B = bars_at(sbase + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    const int G = (int)(K / kGroup);                    // multiple of 8
    const int PAIRS = G / 2;
    constexpr int GB = kQ4 ? 8 : 4;                      // groups per B stage
    const int num_tiles = kGrouped ? ga.tile_offsets[ga.E] * n_tiles : (int)dense_tiles;
    const int t0 = blockIdx.x, dt = gridDim.x;

    if (tid == 0) {
        for (int i = 0; i < NO; ++i) {
            mbar_init(B.full_a + 8 * i, 1);
            mbar_init(B.full_f16 + 8 * i, CONV_WARPS);
            mbar_init(B.ops_free + 8 * i, 1);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(B.full_b + 8 * i, 1);
            mbar_init(B.empty_b + 8 * i, CONV_WARPS);
        }
        for (int i = 0; i < NP; ++i) {
            mbar_init(B.tfull + 8 * i, 1);
            mbar_init(B.tempty + 8 * i, EPI_WARPS);
        }
        for (int i = 0; i < NSC; ++i) {
            mbar_init(B.full_sc + 8 * i, 1);
            mbar_init(B.empty_sc + 8 * i, EPI_WARPS);
        }
        mbar_init(B.drain, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == PROD_WARP && lane == 0) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
        tma_prefetch_desc(&map_dx);
        tma_prefetch_desc(&map_dw);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == PROD_WARP) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int64_t ia = 0, ib = 0, isc = 0;      // stages issued so far (run on across tiles)
            bool ok = true;
            for (int t = t0; t < num_tiles && ok; t += dt) {
                const Tile T = tile_at<kGrouped>(t, M, G, ga, n_tiles);
                // issue in the order the stages are first needed
                for (int g = 0; g < G && ok; ++g) {
                    if (g % SCG == 0) {
                        const int slot = (int)(isc % NSC);
                        if (!(ok = wait_bar<false>(B.empty_sc + 8 * slot, ((isc / NSC) & 1) ^ 1, abort))) break;
                        const uint32_t dst = sbase + OFF_SC + slot * SC_STAGE;
                        mbar_expect_tx(B.full_sc + 8 * slot, SC_STAGE);
                        // dense: dx transposed (x = first row, a multiple of 128);
                        // grouped: dx row-major (segment starts are arbitrary rows)
                        if constexpr (kGrouped)
                            tma_load_2d(dst, &map_dx, g, (int32_t)T.m0, B.full_sc + 8 * slot);
                        else
                            tma_load_2d(dst, &map_dx, (int32_t)T.m0, g, B.full_sc + 8 * slot);
                        tma_load_2d(dst + SC_DX, &map_dw, (int32_t)T.n0, (int32_t)(T.sg0 + g),
                                    B.full_sc + 8 * slot);
                        ++isc;
                    }
                    if (g % GB == 0) {
                        const int slot = (int)(ib % NB);
                        if (!(ok = wait_bar<false>(B.empty_b + 8 * slot, ((ib / NB) & 1) ^ 1, abort))) break;
                        mbar_expect_tx(B.full_b + 8 * slot, B_STAGE);
                        tma_load_2d(sbase + OFF_B + slot * B_STAGE, &map_b, (g / GB) * 128,
                                    (int32_t)T.bn0, B.full_b + 8 * slot);
                        ++ib;
                    }
                    if (g % GA == 0) {
                        const int slot = (int)(ia % NO);
                        if (!(ok = wait_bar<false>(B.ops_free + 8 * slot, ((ia / NO) & 1) ^ 1, abort))) break;
                        mbar_expect_tx(B.full_a + 8 * slot, A_STAGE);
                        tma_load_2d(sbase + OFF_A + slot * A_STAGE, &map_a, g * 32, (int32_t)T.m0,
                                    B.full_a + 8 * slot);
                        ++ia;
                    }
                }
            }
            if (!ok) {
                for (int64_t s = ia - NO; s < ia; ++s)
                    if (s >= 0) drain_wait(B.full_a + 8 * (s % NO), (s / NO) & 1);
                for (int64_t s = ib - NB; s < ib; ++s)
                    if (s >= 0) drain_wait(B.full_b + 8 * (s % NB), (s / NB) & 1);
                for (int64_t s = isc - NSC; s < isc; ++s)
                    if (s >= 0) drain_wait(B.full_sc + 8 * (s % NSC), (s / NSC) & 1);
            }
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool issued_any = false, ok = true;
            uint32_t p = 0;                                 // pair counter (A stage = pair)
            for (int t = t0; t < num_tiles && ok; t += dt) {
                for (int pl = 0; pl < PAIRS; ++pl, ++p) {
                    const int so = (int)(p % NO), ps = (int)(p % NP);
                    const uint32_t po = (uint32_t)((p / NO) & 1), pp = (uint32_t)((p / NP) & 1);
                    // the three probes go out back to back; one branch on all of them
                    const bool ready = mbar_try_wait(B.full_a + 8 * so, po) &
                                       mbar_try_wait(B.full_f16 + 8 * so, po) &
                                       mbar_try_wait(B.tempty + 8 * ps, pp ^ 1);
                    if (!ready) {
                        if (!(ok = wait_bar<false>(B.full_a + 8 * so, po, abort))) break;
                        if (!(ok = wait_bar<false>(B.full_f16 + 8 * so, po, abort))) break;
                        if (!(ok = wait_bar<false>(B.tempty + 8 * ps, pp ^ 1, abort))) break;
                    }
                    tc_fence_after();
                    const uint32_t a_s = sbase + OFF_A + so * A_STAGE;
                    const uint32_t b_s = sbase + OFF_F16 + so * F16_PAIR;
                    const uint32_t d = tmem_base + (uint32_t)(ps * 2 * BN);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            mma_f16(d + h * BN, smem_desc_sw128(a_s + h * 64 + j * 32),
                                    smem_desc_noswizzle(b_s + h * F16_B + j * 256, 128, 512), IDESC, j);
                    mma_commit(B.tfull + 8 * ps);
                    mma_commit(B.ops_free + 8 * so);
                    issued_any = true;
                }
            }
            if (*abort && issued_any) {
                mma_commit(B.drain);
                drain_wait(B.drain, 0);
            }
        }
    } else if (warp >= CONV_WARP0) {
        // ------------------------------------------------------------ converters
        const int ct = tid - CONV_WARP0 * 32;
        uint32_t p = 0, sb = 0;                             // run on across tiles
        bool ok = true;
        for (int t = t0; t < num_tiles && ok; t += dt) {
            for (int pl = 0; pl < PAIRS && ok; ++pl, ++p) {
                const int g0 = 2 * pl;
                if (g0 % GB == 0 && !(ok = wait_bar<true>(B.full_b + 8 * (sb % NB), (sb / NB) & 1, abort))) break;
                // the operand slot is free once the MMAs of pair p - NO completed
                const int so = (int)(p % NO);
                if (!(ok = wait_bar<true>(B.ops_free + 8 * so, (uint32_t)(((p / NO) & 1) ^ 1), abort))) break;
                const uint8_t* src = smem + OFF_B + (sb % NB) * B_STAGE;
                uint8_t* dst = smem + OFF_F16 + so * F16_PAIR;
                convert_group<kQ4>(src, dst, g0 % GB, ct);
                convert_group<kQ4>(src, dst + F16_B, (g0 + 1) % GB, ct);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(B.full_f16 + 8 * so);
                    if ((g0 + 1) % GB == GB - 1) mbar_arrive(B.empty_b + 8 * (sb % NB));
                }
                if ((g0 + 1) % GB == GB - 1) ++sb;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                             // TMEM lane quarter
        const int row = q * 32 + lane;
        const int cb = (warp >> 2) * 32;                    // 32 columns per warp
        uint32_t p = 0, sc = 0;
        bool ok = true;
        for (int t = t0; t < num_tiles && ok; t += dt) {
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.f;
            for (int pl = 0; pl < PAIRS; ++pl, ++p) {
                const int g0 = 2 * pl, ps = (int)(p % NP);
                const int slot = (int)(sc % NSC);
                if (g0 % SCG == 0 && !(ok = wait_bar<true>(B.full_sc + 8 * slot, (sc / NSC) & 1, abort))) break;
                if (!(ok = wait_bar<true>(B.tfull + 8 * ps, (uint32_t)((p / NP) & 1), abort))) break;
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ps * 2 * BN + cb);
                const uint8_t* st = smem + OFF_SC + slot * SC_STAGE;
                float2 dxv;
                if constexpr (kGrouped) {
                    dxv = *reinterpret_cast<const float2*>(reinterpret_cast<const float*>(st) +
                                                           row * SCG + (g0 % SCG));
                } else {                                    // contiguous over the warp's rows
                    const float* dxt = reinterpret_cast<const float*>(st) + (g0 % SCG) * BM + row;
                    dxv = make_float2(dxt[0], dxt[BM]);
                }
                const float* dw0 = reinterpret_cast<const float*>(st + SC_DX) + (g0 % SCG) * BN + cb;
                // the two groups of the pair one after the other (32 partials live);
                // the other warps on this SMSP cover the TMEM latency
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t sv[32];
                    tmem_ld32(taddr + h * BN, sv);
                    tmem_wait_ld();
                    if (h == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(B.tempty + 8 * ps);
                    }
                    const float dh = h ? dxv.y : dxv.x;
                    const float* dwh = dw0 + h * BN;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 w = *reinterpret_cast<const float4*>(dwh + i * 4);
                        acc[4 * i + 0] = fmaf(__uint_as_float(sv[4 * i + 0]), dh * w.x, acc[4 * i + 0]);
                        acc[4 * i + 1] = fmaf(__uint_as_float(sv[4 * i + 1]), dh * w.y, acc[4 * i + 1]);
                        acc[4 * i + 2] = fmaf(__uint_as_float(sv[4 * i + 2]), dh * w.z, acc[4 * i + 2]);
                        acc[4 * i + 3] = fmaf(__uint_as_float(sv[4 * i + 3]), dh * w.w, acc[4 * i + 3]);
                    }
                }
                if ((g0 + 1) % SCG == SCG - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B.empty_sc + 8 * slot);
                    ++sc;
                }
            }
            if (!ok) break;
            const Tile T = tile_at<kGrouped>(t, M, G, ga, n_tiles);
            if (row < T.rows) {
                int64_t orow;
                if constexpr (kGrouped) orow = ga.perm[T.m0 + row];
                else orow = T.m0 + row;
                float* yr = y + orow * ldy + T.n0 + cb;
                const int64_t ncols = N - (T.n0 + cb);
                if (vec4 && ncols >= 32) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float4*>(yr + 4 * i) =
                            make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < ncols) yr[i] = acc[i];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---- pre-pass: int8 codes -> binary16 (optionally gathered) ---------------------------

// Dense: a16[r] = fp16(qx[r]).  Grouped (perm != nullptr): sorted position i
// takes activation row x_row(perm[i]); its scales are gathered into dxg too.
__global__ void __launch_bounds__(256)
widen_rows_kernel(const int8_t* __restrict__ qx, const float* __restrict__ dx, int64_t rows,
                  int64_t K, __half* __restrict__ a16, float* __restrict__ dxg,
                  const int32_t* __restrict__ perm, const int32_t* __restrict__ n_rows,
                  int32_t topk, int32_t x_row_mode) {
    const int64_t chunks = K / 16;                   // 16 codes per thread step
    const int64_t G = K / kGroup;
    const int64_t limit = n_rows ? (int64_t)*n_rows : rows;
    const int64_t total = limit * chunks;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / chunks, c = i % chunks;
        int64_t src = r;
        if (perm) {
            const int32_t p = perm[r];
            src = x_row_mode ? p : p / topk;
        }
        const uint4 v = *reinterpret_cast<const uint4*>(qx + src * K + c * 16);
        uint4 lo, hi;
        s8x16_to_h16(v, lo, hi);
        uint4* o = reinterpret_cast<uint4*>(a16 + r * K + c * 16);
        o[0] = lo;
        o[1] = hi;
        if (dxg && c % 2 == 0) dxg[r * G + c / 2] = dx[src * G + c / 2];
    }
}

// dwT[r][n] = float(dw[n][g]) with r = e * G + g: the scale plane transposed to
// group-major binary32 rows of ldt columns, the layout the epilogue reads.
__global__ void __launch_bounds__(256)
transpose_scales_kernel(const uint16_t* __restrict__ dw, int64_t rows_n, int64_t G, int64_t E,
                        float* __restrict__ dwt, int64_t ldt) {
    const int64_t total = E * rows_n * G;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        // i walks dwT in order: e, g, n (coalesced writes)
        const int64_t n = i % rows_n, eg = i / rows_n;
        const int64_t g = eg % G, e = eg / G;
        dwt[eg * ldt + n] = half_bits_to_float(dw[(e * rows_n + n) * G + g]);
    }
}

// dxt[g][m] = dx[m][g]: activation scales transposed to group-major rows of
// ldm columns, so the epilogue's 32 rows of one group are contiguous.
__global__ void __launch_bounds__(256)
transpose_dx_kernel(const float* __restrict__ dx, int64_t M, int64_t G, float* __restrict__ dxt,
                    int64_t ldm) {
    const int64_t total = M * G;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i % M, g = i / M;               // writes coalesced along m
        dxt[g * ldm + m] = dx[m * G + g];
    }
}

// ---- host side ----------------------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle sw) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of one product: A binary16 [rows][K], B codes [brows][K or K/2],
// dx [rows][G], transposed scales dwT [E*G][ldt] (binary32, n columns used).
// ldm > 0: dx is the transposed plane dxt [G][ldm]; ldm == 0: dx is [rows][G].
bool make_maps(CUtensorMap* ma, CUtensorMap* mb, CUtensorMap* mdx, CUtensorMap* mdw,
               const void* a16, const void* qw, const float* dx, const float* dwt,
               int64_t rows, int64_t brows, int64_t n, int64_t ldt, int64_t sgrows, int64_t K,
               bool q4, int64_t ldm) {
    const int64_t G = K / kGroup;
    const int64_t wbytes = q4 ? K / 2 : K;
    const bool dx_ok = ldm > 0
        ? make_map(mdx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dx, rows, G, ldm * 4, BM, SCG,
                   CU_TENSOR_MAP_SWIZZLE_NONE)
        : make_map(mdx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dx, G, rows, G * 4, SCG, BM,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!dx_ok) return false;
    return make_map(ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a16, K, rows, K * 2, 64, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, wbytes, brows, wbytes, 128, BN,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(mdw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dwt, n, sgrows, ldt * 4, BN, SCG,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <bool kQ4, bool kGrouped>
cudaError_t launch_kernel(dim3 grid, const CUtensorMap& ma, const CUtensorMap& mb,
                          const CUtensorMap& mdx, const CUtensorMap& mdw, float* y, int64_t M,
                          int64_t N, int64_t K, int64_t ldy, GroupedArgs ga, int n_tiles,
                          int64_t dense_tiles, cudaStream_t s) {
    cudaError_t e = ensure_smem_attr((const void*)tc_gemm_kernel<kQ4, kGrouped>, SMEM_BYTES,
                                     9 + (kQ4 ? 1 : 0) + (kGrouped ? 2 : 0));
    if (e != cudaSuccess) return e;
    const bool vec4 = ((uintptr_t)y % 16 == 0) && (ldy % 4 == 0);
    tc_gemm_kernel<kQ4, kGrouped><<<grid, THREADS, SMEM_BYTES, s>>>(ma, mb, mdx, mdw, y, M, N, K,
                                                                    ldy, vec4, ga, n_tiles,
                                                                    dense_tiles);
    return cudaGetLastError();
}

int widen_grid(int64_t work) {
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

size_t align16(size_t v) { return (v + 15) / 16 * 16; }

}  // namespace

int tc_tile_m() { return BM; }

bool tc_gemm_supported(int64_t M, int64_t N, int64_t K, const void* dx, const void* dw) {
    (void)M; (void)N;
    return K % 256 == 0 && ((uintptr_t)dx % 16 == 0) && ((uintptr_t)dw % 16 == 0) &&
           encoder() != nullptr;
}

int64_t ldt_of(int64_t N) { return (N + 3) / 4 * 4; }

// dense workspace: a16 [M][K] binary16 | dwT [G][ldt(N)] binary32 | dxT [G][ldt(M)] binary32
size_t tc_gemm_workspace(int64_t M, int64_t N, int64_t K) {
    const int64_t G = K / kGroup;
    return align16((size_t)M * K * 2) + align16((size_t)G * ldt_of(N) * 4) +
           align16((size_t)G * ldt_of(M) * 4);
}

cudaError_t launch_tc_gemm(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                           const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                           void* workspace, cudaStream_t s) {
    const int64_t G = K / kGroup, ldt = ldt_of(N), ldm = ldt_of(M);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    __half* a16 = reinterpret_cast<__half*>(ws);
    float* dwt = reinterpret_cast<float*>(ws + align16((size_t)M * K * 2));
    float* dxt = reinterpret_cast<float*>(ws + align16((size_t)M * K * 2) + align16((size_t)G * ldt * 4));
    widen_rows_kernel<<<widen_grid(M * (K / 16)), 256, 0, s>>>(qx, dx, M, K, a16, nullptr, nullptr,
                                                               nullptr, 1, 0);
    transpose_scales_kernel<<<widen_grid(N * G), 256, 0, s>>>(dw, N, G, 1, dwt, ldt);
    transpose_dx_kernel<<<widen_grid(M * G), 256, 0, s>>>(dx, M, G, dxt, ldm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb, mdx, mdw;
    if (!make_maps(&ma, &mb, &mdx, &mdw, a16, qw, dxt, dwt, M, N, N, ldt, G, K, q4, ldm))
        return cudaErrorInvalidValue;
    const int n_tiles = (int)((N + BN - 1) / BN);
    const int64_t tiles = (int64_t)n_tiles * ((M + BM - 1) / BM);
    const int64_t ctas = tiles < sm_count() ? tiles : sm_count();
    dim3 grid((unsigned)ctas);
    GroupedArgs ga{};
    return q4 ? launch_kernel<true, false>(grid, ma, mb, mdx, mdw, y, M, N, K, ldy, ga, n_tiles, tiles, s)
              : launch_kernel<false, false>(grid, ma, mb, mdx, mdw, y, M, N, K, ldy, ga, n_tiles, tiles, s);
}

// MoE workspace after the routing tables: a16 [P][K] binary16, dxg [P][G]
// binary32 (gathered activation rows and scales in expert order) and the
// transposed scales dwT [E*G][ldt] binary32.
size_t tc_grouped_workspace(int64_t P, int64_t N, int64_t K, int32_t E) {
    const int64_t G = K / kGroup;
    return align16((size_t)P * K * 2) + align16((size_t)P * G * 4) +
           align16((size_t)E * G * ldt_of(N) * 4);
}

cudaError_t launch_tc_grouped(const int8_t* qx, const float* dx, int64_t P, int64_t N, int64_t K,
                              const uint8_t* qw4, const uint16_t* dw, float* y, int32_t E,
                              int32_t topk, int32_t x_row_mode, const int32_t* perm,
                              const int32_t* offsets, const int32_t* tile_offsets,
                              void* workspace, cudaStream_t s) {
    const int64_t G = K / kGroup, ldt = ldt_of(N);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    __half* a16 = reinterpret_cast<__half*>(ws);
    float* dxg = reinterpret_cast<float*>(ws + align16((size_t)P * K * 2));
    float* dwt = reinterpret_cast<float*>(ws + align16((size_t)P * K * 2) + align16((size_t)P * G * 4));
    // gather + widen the routed rows (count read on the device: offsets[E])
    widen_rows_kernel<<<widen_grid(P * (K / 16)), 256, 0, s>>>(qx, dx, P, K, a16, dxg, perm,
                                                               offsets + E, topk, x_row_mode);
    transpose_scales_kernel<<<widen_grid((int64_t)E * N * G), 256, 0, s>>>(dw, N, G, E, dwt, ldt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb, mdx, mdw;
    if (!make_maps(&ma, &mb, &mdx, &mdw, a16, qw4, dxg, dwt, P, (int64_t)E * N, N, ldt,
                   (int64_t)E * G, K, true, 0))
        return cudaErrorInvalidValue;
    const int n_tiles = (int)((N + BN - 1) / BN);
    GroupedArgs ga{perm, offsets, tile_offsets, E, N};
    dim3 grid((unsigned)sm_count());
    return launch_kernel<true, true>(grid, ma, mb, mdx, mdw, y, P, N, K, N, ga, n_tiles, 0, s);
}

unsigned int read_and_clear_tc_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    cudaMemcpyToSymbol(g_tc_error, &z, sizeof z);
    return v;
}

}  // namespace qg
