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
// Per CTA (persistent, one per SM; 576 threads dense, 768 MoE): 128 x 128
// output tiles, K walked one pair of 32-groups at a time.
//   pre-pass    activation codes widened to binary16 once per call (for the
//               MoE product also gathered into expert order with their
//               scales); dense: the weight codes widened to binary16 too and
//               the weight scales transposed to group-major binary32, all
//               three in one launch.  Each kernel of a call is a programmatic
//               dependent launch of the one before.
//   warp 16     TMA producer: binary16 A stages (one pair of groups, 128-byte
//               swizzle, the operand layout the MMA reads directly); dense:
//               a binary16 B stage of the same form on the same barrier, and
//               the dx / dw scale stages every 8 groups.
//   warps 18-19 (MoE only) TMA producers of the packed 4-bit B stages (8
//               groups, 128-byte swizzle) and of the scale stages, each on its
//               own thread so that no stream waits behind another's ring.
//   warps 20-23 (MoE only) converters, one B row per thread: 4-bit codes ->
//               binary16 into the canonical K-major no-swizzle layout (8 x
//               16-byte core matrices), a pair of groups per operand slot.
//   warp 17     one thread issues, per pair, four K=16 MMAs (two per group,
//               the first of each overwrites) into one of two 256-column TMEM
//               pair slots and one commit.
//   warps 0-15  epilogue: 16-lane x 256-bit TMEM reads, the pair slot is
//               released as soon as it is read, then y += (S * dw) * dx on
//               packed f32x2 instructions into binary32 registers.
// Dense tail split: when the tile count leaves the grid's last round partly
// empty, those last tiles are cut along K into chunks (multiples of 8 groups)
// that fill the round; each chunk stores binary32 partial sums and a small
// kernel adds each tile's chunks in chunk order.
// Every mbarrier wait is bounded; on a timeout the CTA sets a device error
// word, drains its own TMA copies and MMAs, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace qg {

__device__ unsigned int g_tc_error = 0;
// Cycles a pipeline wait may last before the kernel gives up (~2 s at 2 GHz);
// lowered only by the test-only qg_debug_set_wait_limit.
constexpr long long kWaitCycles = 4000000000ll;
__device__ long long g_wait_limit = kWaitCycles;

namespace {

using namespace tc;

constexpr int BM = 128, BN = 128;
constexpr int GA = 2;                  // groups per A stage = one pair (64 binary16 = 128-byte rows)
constexpr int NO = 4;                  // operand slots: binary16 A stage + binary16 B pair
constexpr int NB = 4;                  // B code stages (each 128-byte rows: 4 Q8 / 8 Q4 groups)
constexpr int NP = 2;                  // TMEM pair slots (two 128-column accumulators each)
constexpr int NPMAX = 8;               // MoE pair slots at most (narrow tiles: 8 x 2 x 32 columns)
constexpr int SCG = 8;                 // groups per scale stage
constexpr int NSC = 4;                 // scale stages
constexpr int EPI_WARPS = 16;          // 4 per TMEM lane quarter, 32 columns each
constexpr int PROD_WARP = 16, MMA_WARP = 17, BPROD_WARP = 18, SPROD_WARP = 19;
constexpr int CONV_WARP0 = 20, CONV_WARPS = 4;
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int THREADS = (CONV_WARP0 + CONV_WARPS) * 32;   // 768 (MoE): 80 registers a thread
constexpr int THREADS_DENSE = (MMA_WARP + 1) * 32;         // 576 (dense: warps 0-17 only): 96
static_assert(MMA_WARP + 1 == 18 && PROD_WARP < MMA_WARP && EPI_WARPS == PROD_WARP,
              "the dense kernel launches epilogue, producer and MMA warps only");

constexpr int A_STAGE = BM * 128;                    // 16384
constexpr int B_STAGE = BN * 128;                    // 16384
constexpr int F16_B = BN * 32 * 2;                   // 8192: one group of binary16 B
constexpr int F16_PAIR = 2 * F16_B;                  // 16384
// scale stage: dx [128 rows][8 groups] f32, then dw: dense [8 groups][128
// columns] f32 (permuted), MoE [128 rows][8 groups] binary16.
constexpr int SC_DX = BM * SCG * 4;                  // 4096
constexpr int SC_DW = SCG * BN * 4;                  // 4096
constexpr int SC_STAGE = SC_DX + SC_DW;              // 8192
constexpr int SC_DW16 = BN * SCG * 2;                // 2048: MoE dw

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + NO * A_STAGE;
constexpr int OFF_F16 = OFF_B + NB * B_STAGE;
constexpr int OFF_SC = OFF_F16 + NO * F16_PAIR;
constexpr int OFF_BAR = OFF_SC + NSC * SC_STAGE;
constexpr int NUM_BARS = 3 * NO + 2 * NB + 2 * NPMAX + 2 * NSC + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;     // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_B % 1024 == 0 && OFF_F16 % 1024 == 0, "swizzled stages need 1 KiB alignment");

constexpr uint32_t TMEM_COLS = NP * 2 * BN;          // 512: two pair slots of two groups
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
constexpr uint32_t kSpinLimit = 1u << 22;          // drain polls after an abort
constexpr uint32_t kSleepHintNs = 20000;             // a waiter sleeps until the phase flips

// full_a: the TMA A stage landed (dense: with the binary16 B stage, so both
// operands of the slot are ready); full_ops (MoE): the converters saw full_a
// and wrote the binary16 B pair, so both operands are ready; done: the
// MMAs of the pair completed (one commit: operand slot free and the pair's
// accumulators readable); tempty: the epilogue has read the TMEM pair slot;
// afull (MoE tiles): the MMAs into a TMEM pair slot completed.
struct Bars {
    uint32_t full_a, full_ops, done, full_b, empty_b, tempty, afull, full_sc, empty_sc, drain;
};

__device__ __forceinline__ Bars bars_at(uint32_t base) {
    Bars b;
    b.full_a = base;
    b.full_ops = b.full_a + 8 * NO;
    b.done = b.full_ops + 8 * NO;
    b.full_b = b.done + 8 * NO;
    b.empty_b = b.full_b + 8 * NB;
    b.tempty = b.empty_b + 8 * NB;
    b.afull = b.tempty + 8 * NPMAX;
    b.full_sc = b.afull + 8 * NPMAX;
    b.empty_sc = b.full_sc + 8 * NSC;
    b.drain = b.empty_sc + 8 * NSC;
    return b;
}

// Bounded wait: the thread sleeps in try_wait until the phase completes; after
// g_wait_limit cycles without completion (or when another role gave up) it returns
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
        bool late = clock64() - start > g_wait_limit;
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

// Groups gi, gi + 1 of the packed 4-bit B stage -> the binary16 B pair
// (canonical no-swizzle K-major layout: core matrix (row/8, k8) at
// (row/8)*512 + k8*128, row%8 at +16 each; the second group F16_B further).
// Thread ct owns B row ct; all its shared loads go out before any store.
__device__ __forceinline__ void convert_pair_q4(const uint8_t* src, uint8_t* dst, int gi, int ct) {
    static_assert(CONV_THREADS == BN, "one converter thread per B row");
    const int row = ct, sw = row & 7;
    const uint8_t* srow = src + row * 128;
    uint8_t* drow = dst + (row >> 3) * 512 + sw * 16;
    uint4 v[2];                                        // one 16-byte group each
#pragma unroll
    for (int c = 0; c < 2; ++c)
        v[c] = *reinterpret_cast<const uint4*>(srow + (((gi + c) ^ sw) << 4));
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        // byte j: element j (low nibble), element j+16 (high nibble)
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
        uint32_t lo_h[8], hi_h[8];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t l = w[t] & 0x0f0f0f0fu, h = (w[t] >> 4) & 0x0f0f0f0fu;
            lo_h[2 * t] = u4x2_to_h2(l, 0x4140);
            lo_h[2 * t + 1] = u4x2_to_h2(l, 0x4342);
            hi_h[2 * t] = u4x2_to_h2(h, 0x4140);
            hi_h[2 * t + 1] = u4x2_to_h2(h, 0x4342);
        }
        uint8_t* o = drow + c * F16_B;
        *reinterpret_cast<uint4*>(o) = make_uint4(lo_h[0], lo_h[1], lo_h[2], lo_h[3]);
        *reinterpret_cast<uint4*>(o + 128) = make_uint4(lo_h[4], lo_h[5], lo_h[6], lo_h[7]);
        *reinterpret_cast<uint4*>(o + 256) = make_uint4(hi_h[0], hi_h[1], hi_h[2], hi_h[3]);
        *reinterpret_cast<uint4*>(o + 384) = make_uint4(hi_h[4], hi_h[5], hi_h[6], hi_h[7]);
    }
}

struct GroupedArgs {
    const int32_t* perm;          // sorted position -> pair index
    const int32_t* offsets;       // [E+1]
    const int32_t* tile_offsets;  // [E+1] in 128-row tiles
    const int4* tile_info;        // per 128-row tile: {first sorted row, rows, expert, 0}
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
        const int4 info = ga.tile_info[mt];
        T.m0 = info.x;
        T.rows = info.y;
        T.bn0 = (int64_t)info.z * ga.N + T.n0;
        T.sg0 = (int64_t)info.z * G;
    } else {
        T.m0 = mt * BM;
        T.rows = min64(BM, M - T.m0);
        T.bn0 = T.n0;
        T.sg0 = 0;
    }
    return T;
}

// Dense work units.  Units [0, full) are whole output tiles.  When the tile
// count leaves the last round of the persistent grid partly empty, each of
// those last tiles is cut along K into `split` chunks of equal length (a
// multiple of 8 groups, so every stage boundary stays where it was): unit
// full + l * split + c is chunk c of tile full + l.  A chunk's binary32 sums go
// to partial slot l * split + c of `part` (BM x BN each), and
// tail_reduce_kernel adds a tile's chunks in chunk order into y.
struct TailArgs {
    int full;          // whole-tile units
    int split;         // K chunks per tail tile (1: no tail split)
    float* part;       // [(units - full)][BM][BN] binary32
};

struct Unit {
    int tile, g0, pairs, slot;    // output tile, first group, pairs of groups, partial slot (-1: y)
};

__device__ __forceinline__ Unit unit_at(int t, int PAIRS, const TailArgs& ta) {
    Unit u;
    if (t < ta.full) {
        u.tile = t;
        u.g0 = 0;
        u.pairs = PAIRS;
        u.slot = -1;
    } else {
        const int v = t - ta.full;
        u.pairs = PAIRS / ta.split;
        u.tile = ta.full + v / ta.split;
        u.g0 = 2 * u.pairs * (v % ta.split);
        u.slot = v;
    }
    return u;
}

// Columns a MoE tile's pair slot gives each of its two groups: the tile's
// rows rounded up to 32, 64 or 128 (the MMA N is the rows rounded up to 16).
__device__ __forceinline__ int slot_width(int rows) { return rows <= 32 ? 32 : (rows <= 64 ? 64 : BN); }

// One MoE output tile of the epilogue (the dense epilogue is inline in the
// kernel).  TMEM lanes = weight rows (dw per lane, binary16 as stored),
// columns = the segment's rows (dx per column).  Fragments and arithmetic are
// the dense epilogue's (16-lane x 256-bit reads, y += (S * dw) * dx on packed
// f32x2), but warp w covers its TMEM quarter (w % 4) over CW columns from
// (w / 4) CW, with CW = 8, 16 or 32 taken from the tile's row count (at most
// 32, 64 or 128 columns in use): short segments keep all 16 warps busy on a
// quarter of the reads each instead of leaving 12 idle.  Each output is still
// one thread's running sum over the groups in order.  The pair slots follow
// the MMA issuer's ring: slot r mod (8 / 4 / 2) of 2 x 4 CW columns, waited on
// through its afull barrier (apar: per slot, the parity of its next phase).
// Returns false when a wait gave up.
template <int CW>
__device__ __forceinline__ bool epilogue_tile(const Bars& B, const uint8_t* smem, uint32_t tmem_base,
                                              volatile int* abort, int PAIRS, uint32_t& r, uint32_t& apar,
                                              uint32_t& sc,
                                              int warp, int lane, int t, int trows, int64_t M, int G,
                                              int n_tiles, float* __restrict__ y, int64_t N, int64_t ldy,
                                              const GroupedArgs& ga) {
    constexpr int NJ = CW / 8;                          // 8-column blocks per warp
    constexpr int W = 4 * CW;                           // columns of one group in a slot
    constexpr uint32_t kSlotMask = (uint32_t)(2 * BN / W) - 1;
    const int q = warp & 3;                             // TMEM lane quarter
    const int cb = (warp >> 2) * CW;
    const int c2 = 2 * (lane & 3);
    const int rb = q * 32 + (lane >> 2);                // lanes rb + 8 i, i = 0..3
    // a warp with no valid output (short MoE segments, ragged last tile)
    // keeps the barrier protocol but skips the readout and math
    const bool live = cb < trows;
    uint64_t acc[4][NJ];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < NJ; ++j) acc[i][j] = 0ull;
    for (int pl = 0; pl < PAIRS; ++pl, ++r) {
        const int g0 = 2 * pl, ps = (int)(r & kSlotMask);
        const int slot = (int)(sc % NSC);
        if (g0 % SCG == 0 && !wait_bar<true>(B.full_sc + 8 * slot, (sc / NSC) & 1, abort)) return false;
        // every warp, live or not, waits for the slot's MMAs before releasing it
        if (!wait_bar<true>(B.afull + 8 * ps, (apar >> ps) & 1u, abort)) return false;
        apar ^= 1u << ps;
        tc_fence_after();
        if (live) {
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ps * 2 * W + cb);
            const float* scf = reinterpret_cast<const float*>(smem + OFF_SC + slot * SC_STAGE);
            // per-lane scales of the pair's two groups
            float2 lsc[4];
            const __half2* dws = reinterpret_cast<const __half2*>(smem + OFF_SC + slot * SC_STAGE + SC_DX);
#pragma unroll
            for (int i = 0; i < 4; ++i) lsc[i] = __half22float2(dws[((rb + 8 * i) * SCG + (g0 % SCG)) / 2]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // per-column scale pairs of group g0 + h for the warp's column blocks
                uint64_t csc[NJ];
                const float* dxc = scf + (cb + c2) * SCG + (g0 % SCG) + h;
#pragma unroll
                for (int j = 0; j < NJ; ++j) csc[j] = pack2(dxc[8 * j * SCG], dxc[(8 * j + 1) * SCG]);
                if constexpr (CW == 8) {
                    const uint32_t ta = taddr + h * W;
                    uint32_t s0[4], s1[4];
                    tmem_ld16x256b_x1(ta, s0);                 // lanes rb, rb + 8
                    tmem_ld16x256b_x1(ta + (16u << 16), s1);   // lanes rb + 16, rb + 24
                    tmem_wait_ld();
                    if (h == 1) {                              // pair slot read out
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(B.tempty + 8 * ps);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float d = h ? lsc[i].y : lsc[i].x;
                        const uint32_t* sv = i < 2 ? s0 : s1;
                        const int e = 2 * (i & 1);
                        fma_f32x2(acc[i][0], mul_f32x2(pack2u(sv[e], sv[e + 1]), pack2(d, d)), csc[0]);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < CW / 16; ++k) {        // 16-column halves
                        const uint32_t ta = taddr + h * W + 16 * k;
                        uint32_t s0[8], s1[8];
                        tmem_ld16x256b_x2(ta, s0);             // lanes rb, rb + 8
                        tmem_ld16x256b_x2(ta + (16u << 16), s1);   // lanes rb + 16, rb + 24
                        tmem_wait_ld();
                        if (h == 1 && k == CW / 16 - 1) {      // pair slot read out
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(B.tempty + 8 * ps);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float d = h ? lsc[i].y : lsc[i].x;
                            const uint64_t d2 = pack2(d, d);
                            const uint32_t* sv = i < 2 ? s0 : s1;
                            const int e = 2 * (i & 1);
                            fma_f32x2(acc[i][2 * k], mul_f32x2(pack2u(sv[e], sv[e + 1]), d2), csc[2 * k]);
                            fma_f32x2(acc[i][2 * k + 1], mul_f32x2(pack2u(sv[4 + e], sv[4 + e + 1]), d2), csc[2 * k + 1]);
                        }
                    }
                }
            }
        } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.tempty + 8 * ps);
        }
        if ((g0 + 1) % SCG == SCG - 1) {
            __syncwarp();
            if (lane == 0) mbar_arrive(B.empty_sc + 8 * slot);
            ++sc;
        }
    }
    if (!live) return true;
    const Tile T = tile_at<true>(t, M, G, ga, n_tiles);        // fetched again: fewer live registers
    // lane rb + 8 i = output column n0 + rb + 8 i; column = segment row
#pragma unroll
    for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = cb + 8 * j + c2 + e;
            if (r < T.rows) {
                float* yr = y + (int64_t)ga.perm[T.m0 + r] * ldy + T.n0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 v = unpack2(acc[i][j]);
                    if (T.n0 + rb + 8 * i < N) yr[rb + 8 * i] = e ? v.y : v.x;
                }
            }
        }
    return true;
}

// Persistent: CTA b takes tiles b, b + gridDim.x, ...  All roles walk the same
// tile sequence; ring positions and barrier phases run on across tiles.
template <bool kQ4, bool kGrouped>
__global__ void __launch_bounds__(kGrouped ? THREADS : THREADS_DENSE, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_dx, const __grid_constant__ CUtensorMap map_dw,
               float* __restrict__ y, int64_t M, int64_t N, int64_t K, int64_t ldy, bool vec2,
               GroupedArgs ga, int n_tiles, int64_t dense_tiles, TailArgs ta) {
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
    const int t0 = blockIdx.x, dt = gridDim.x;

    if (tid == 0) {
        for (int i = 0; i < NO; ++i) {
            mbar_init(B.full_a + 8 * i, 1);
            mbar_init(B.full_ops + 8 * i, CONV_WARPS);
            mbar_init(B.done + 8 * i, 1);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(B.full_b + 8 * i, 1);
            mbar_init(B.empty_b + 8 * i, CONV_WARPS);
        }
        for (int i = 0; i < NPMAX; ++i) {
            mbar_init(B.tempty + 8 * i, EPI_WARPS);
            mbar_init(B.afull + 8 * i, 1);
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
    // launched as a programmatic dependent of the pre-pass: barrier setup and the
    // TMEM allocation above overlap its end; everything below may read its output
    pdl_wait();
    const int num_tiles = kGrouped ? ga.tile_offsets[ga.E] * n_tiles : (int)dense_tiles;

    const bool producer = warp == PROD_WARP || (kGrouped && (warp == BPROD_WARP || warp == SPROD_WARP));
    if (producer) {
        // ------------------------------------------------------------ producers
        // Dense: one thread issues every stream.  MoE: one thread per stream
        // (A stages, 4-bit B stages, scale stages), so that no stream waits
        // behind another's ring: the scale stages are released by the
        // epilogue, which runs up to a TMEM ring behind the MMAs.
        if (lane == 0) {
            const bool do_a = warp == PROD_WARP;
            const bool do_b = kGrouped && warp == BPROD_WARP;
            const bool do_sc = !kGrouped || warp == SPROD_WARP;
            int64_t ia = 0, ib = 0, isc = 0;      // stages issued so far (run on across tiles)
            bool ok = true;
            for (int t = t0; t < num_tiles && ok; t += dt) {
                int tile = t, gb = 0, ge = G;
                if constexpr (!kGrouped) {
                    const Unit u = unit_at(t, PAIRS, ta);
                    tile = u.tile;
                    gb = u.g0;
                    ge = u.g0 + 2 * u.pairs;
                }
                const Tile T = tile_at<kGrouped>(tile, M, G, ga, n_tiles);
                // issue in the order the stages are first needed
                for (int g = gb; g < ge && ok; ++g) {
                    if (do_sc && g % SCG == 0) {
                        const int slot = (int)(isc % NSC);
                        if (!(ok = wait_bar<false>(B.empty_sc + 8 * slot, ((isc / NSC) & 1) ^ 1, abort))) break;
                        const uint32_t dst = sbase + OFF_SC + slot * SC_STAGE;
                        mbar_expect_tx(B.full_sc + 8 * slot, kGrouped ? SC_DX + SC_DW16 : SC_STAGE);
                        // dx row-major [rows][G]: x = g, a multiple of 8 groups (32 bytes)
                        tma_load_2d(dst, &map_dx, g, (int32_t)T.m0, B.full_sc + 8 * slot);
                        if constexpr (kGrouped)        // dw binary16 [E*N][G] as stored: x = g (16 bytes)
                            tma_load_2d(dst + SC_DX, &map_dw, g, (int32_t)T.bn0, B.full_sc + 8 * slot);
                        else                           // dwT binary32 [G][ldt], permuted columns
                            tma_load_2d(dst + SC_DX, &map_dw, (int32_t)T.n0, (int32_t)(T.sg0 + g),
                                        B.full_sc + 8 * slot);
                        ++isc;
                    }
                    if (do_b && g % GB == 0) {
                        const int slot = (int)(ib % NB);
                        if (!(ok = wait_bar<false>(B.empty_b + 8 * slot, ((ib / NB) & 1) ^ 1, abort))) break;
                        mbar_expect_tx(B.full_b + 8 * slot, B_STAGE);
                        tma_load_2d(sbase + OFF_B + slot * B_STAGE, &map_b, (g / GB) * 128,
                                    (int32_t)T.bn0, B.full_b + 8 * slot);
                        ++ib;
                    }
                    if (do_a && g % GA == 0) {
                        const int slot = (int)(ia % NO);
                        if (!(ok = wait_bar<false>(B.done + 8 * slot, ((ia / NO) & 1) ^ 1, abort))) break;
                        mbar_expect_tx(B.full_a + 8 * slot, kGrouped ? A_STAGE : A_STAGE + F16_PAIR);
                        tma_load_2d(sbase + OFF_A + slot * A_STAGE, &map_a, g * 32, (int32_t)T.m0,
                                    B.full_a + 8 * slot);
                        if constexpr (!kGrouped)       // binary16 weights [N][K]: the pair's 64 columns
                            tma_load_2d(sbase + OFF_F16 + slot * F16_PAIR, &map_b, g * 32,
                                        (int32_t)T.bn0, B.full_a + 8 * slot);
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
            if constexpr (kGrouped) {
                // MoE tiles put the 128 weight rows on the MMA's M side (TMEM
                // lanes) and the segment's rows on N, rounded up to 16: short
                // segments cost short MMAs.  A tile of at most W = 32 / 64 / 128
                // columns packs 8 / 4 / 2 pair slots (2 x W columns each) into
                // the 512 TMEM columns, so the MMAs run up to that many pairs
                // ahead of the epilogue.  The epilogue waits on the slot's own
                // afull barrier (never more than one phase ahead: a slot is
                // reused only after tempty); when W changes, every slot of the
                // old layout is read out before the new layout is written.
                uint32_t tpar = 0;                          // per slot: parity of its uses so far
                uint32_t r = 0;                             // ring position in the current layout
                int width = 0;
                int next_rows = t0 < num_tiles ? tile_at<kGrouped>(t0, M, G, ga, n_tiles).rows : BM;
                for (int t = t0; t < num_tiles && ok; t += dt) {
                    const int rows = next_rows;
                    if (t + dt < num_tiles) next_rows = tile_at<kGrouped>(t + dt, M, G, ga, n_tiles).rows;
                    const int nt = min(BM, max(16, (rows + 15) & ~15));
                    const uint32_t idesc = idesc_f16_f32(BN, nt);
                    const int W = slot_width(rows);
                    if (W != width) {
                        for (int b = 0; b < NPMAX && ok; ++b)
                            ok = wait_bar<false>(B.tempty + 8 * b, ((tpar >> b) & 1u) ^ 1u, abort);
                        if (!ok) break;
                        width = W;
                        r = 0;
                    }
                    const uint32_t nps_mask = (uint32_t)(2 * BN / W) - 1;   // 8, 4 or 2 slots
                    for (int pl = 0; pl < PAIRS; ++pl, ++p, ++r) {
                        const int so = (int)(p % NO), b = (int)(r & nps_mask);
                        const uint32_t po = (uint32_t)((p / NO) & 1), tp = ((tpar >> b) & 1u) ^ 1u;
                        const bool ready = mbar_try_wait(B.full_ops + 8 * so, po) &
                                           mbar_try_wait(B.tempty + 8 * b, tp);
                        if (!ready) {
                            if (!(ok = wait_bar<false>(B.full_ops + 8 * so, po, abort))) break;
                            if (!(ok = wait_bar<false>(B.tempty + 8 * b, tp, abort))) break;
                        }
                        tc_fence_after();
                        const uint32_t a_s = sbase + OFF_A + so * A_STAGE;
                        const uint32_t b_s = sbase + OFF_F16 + so * F16_PAIR;
                        const uint32_t d = tmem_base + (uint32_t)(b * 2 * W);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const uint64_t da = smem_desc_sw128(a_s + h * 64 + j * 32);
                                const uint64_t db = smem_desc_noswizzle(b_s + h * F16_B + j * 256, 128, 512);
                                mma_f16(d + h * W, db, da, idesc, j);
                            }
                        mma_commit(B.done + 8 * so);
                        mma_commit(B.afull + 8 * b);
                        tpar ^= 1u << b;
                        issued_any = true;
                    }
                }
            } else {
                for (int t = t0; t < num_tiles && ok; t += dt) {
                    const int np = unit_at(t, PAIRS, ta).pairs;
                    for (int pl = 0; pl < np; ++pl, ++p) {
                        const int so = (int)(p % NO), ps = (int)(p % NP);
                        const uint32_t po = (uint32_t)((p / NO) & 1), pp = (uint32_t)((p / NP) & 1);
                        // both probes go out back to back; one branch on the pair
                        const bool ready = mbar_try_wait(B.full_a + 8 * so, po) &
                                           mbar_try_wait(B.tempty + 8 * ps, pp ^ 1);
                        if (!ready) {
                            if (!(ok = wait_bar<false>(B.full_a + 8 * so, po, abort))) break;
                            if (!(ok = wait_bar<false>(B.tempty + 8 * ps, pp ^ 1, abort))) break;
                        }
                        tc_fence_after();
                        const uint32_t a_s = sbase + OFF_A + so * A_STAGE;
                        const uint32_t b_s = sbase + OFF_F16 + so * F16_PAIR;
                        const uint32_t d = tmem_base + (uint32_t)(ps * 2 * BN);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const uint64_t da = smem_desc_sw128(a_s + h * 64 + j * 32);
                                const uint64_t db = smem_desc_sw128(b_s + h * 64 + j * 32);
                                mma_f16(d + h * BN, da, db, IDESC, j);
                            }
                        mma_commit(B.done + 8 * so);
                        issued_any = true;
                    }
                }
            }
            if (*abort && issued_any) {
                mma_commit(B.drain);
                drain_wait(B.drain, 0);
            }
        }
    } else if (warp >= CONV_WARP0) {
      // -------------------------------------------------------------- converters (MoE;
      // the dense kernel is launched without these warps)
      if constexpr (kGrouped) {
        static_assert(kQ4, "the MoE weights are 4-bit");
        const int ct = tid - CONV_WARP0 * 32;
        uint32_t p = 0, sb = 0;                             // run on across tiles
        bool ok = true;
        for (int t = t0; t < num_tiles && ok; t += dt) {
            for (int pl = 0; pl < PAIRS && ok; ++pl, ++p) {
                const int g0 = 2 * pl;
                if (g0 % GB == 0 && !(ok = wait_bar<true>(B.full_b + 8 * (sb % NB), (sb / NB) & 1, abort))) break;
                // the operand slot is free once the MMAs of pair p - NO completed
                const int so = (int)(p % NO);
                if (!(ok = wait_bar<true>(B.done + 8 * so, (uint32_t)(((p / NO) & 1) ^ 1), abort))) break;
                const uint8_t* src = smem + OFF_B + (sb % NB) * B_STAGE;
                uint8_t* dst = smem + OFF_F16 + so * F16_PAIR;
                convert_pair_q4(src, dst, g0 % GB, ct);
                fence_proxy_async_smem();
                // the A stage of the slot has landed too: full_ops then stands for both
                if (!(ok = wait_bar<true>(B.full_a + 8 * so, (uint32_t)((p / NO) & 1), abort))) break;
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(B.full_ops + 8 * so);
                    if ((g0 + 1) % GB == GB - 1) mbar_arrive(B.empty_b + 8 * (sb % NB));
                }
                if ((g0 + 1) % GB == GB - 1) ++sb;
            }
        }
      }
    } else {
        // ------------------------------------------------------------ epilogue
        if constexpr (kGrouped) {
            // MoE tiles: columns per warp from the segment's row count
            uint32_t r = 0, apar = 0, sc = 0;
            int width = 0;
            for (int t = t0; t < num_tiles; t += dt) {
                const int trows = (int)tile_at<kGrouped>(t, M, G, ga, n_tiles).rows;
                const int W = slot_width(trows);
                if (W != width) {                           // the issuer restarts its ring too
                    width = W;
                    r = 0;
                }
                bool ok;
                if (W == 32)
                    ok = epilogue_tile<8>(B, smem, tmem_base, abort, PAIRS, r, apar, sc, warp, lane, t, trows, M, G, n_tiles, y, N, ldy, ga);
                else if (W == 64)
                    ok = epilogue_tile<16>(B, smem, tmem_base, abort, PAIRS, r, apar, sc, warp, lane, t, trows, M, G, n_tiles, y, N, ldy, ga);
                else
                    ok = epilogue_tile<32>(B, smem, tmem_base, abort, PAIRS, r, apar, sc, warp, lane, t, trows, M, G, n_tiles, y, N, ldy, ga);
                if (!ok) break;
            }
        } else {
            // Dense tiles.  TMEM is read in 16-lane x 256-bit fragments: per
            // 8-column block a thread holds 2 adjacent columns of 2 lanes (8
            // apart), so each scale pair serves 2 partials, and the column pairs
            // go through packed f32x2 multiplies and FMAs.  Warp w covers the 32
            // lanes of its TMEM quarter (w % 4) and 32 columns.  Lanes = A rows
            // (dx per lane), columns = B rows (dw per column; the dw stage holds
            // each 32-column block permuted so that a thread's 8 columns are
            // contiguous: 2 x 16-byte loads a group).  y += (S * dw) * dx, the
            // roundings of the MoE epilogue.
            const int q = warp & 3;                             // TMEM lane quarter
            const int cb = (warp >> 2) * 32;                    // 32 columns per warp
            const int c2 = 2 * (lane & 3);
            const int rb = q * 32 + (lane >> 2);                // lanes rb + 8 i, i = 0..3
            uint32_t p = 0, sc = 0;
            bool ok = true;
            for (int t = t0; t < num_tiles && ok; t += dt) {
                // a warp with no valid output (ragged last tile) keeps the
                // barrier protocol but skips the readout and math
                const Unit u = unit_at(t, PAIRS, ta);
                const int trows = (int)tile_at<kGrouped>(u.tile, M, G, ga, n_tiles).rows;
                const bool live = q * 32 < trows;
                uint64_t acc[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = 0ull;
                for (int pl = 0; pl < u.pairs; ++pl, ++p) {
                    const int g0 = 2 * pl, ps = (int)(p % NP), so = (int)(p % NO);
                    const int slot = (int)(sc % NSC);
                    if (g0 % SCG == 0 && !(ok = wait_bar<true>(B.full_sc + 8 * slot, (sc / NSC) & 1, abort))) break;
                    if (!(ok = wait_bar<true>(B.done + 8 * so, (uint32_t)((p / NO) & 1), abort))) break;
                    tc_fence_after();
                    if (live) {
                        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                                               (uint32_t)(ps * 2 * BN + cb);
                        const float* scf = reinterpret_cast<const float*>(smem + OFF_SC + slot * SC_STAGE);
                        // per-lane scales of the pair's two groups
                        float2 lsc[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            lsc[i] = *reinterpret_cast<const float2*>(scf + (rb + 8 * i) * SCG + (g0 % SCG));
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // per-column scale pairs of group g0 + h for column blocks 0..3
                            uint64_t csc[4];
                            const float* dwp = scf + SC_DX / 4 + ((g0 % SCG) + h) * BN + cb + 4 * c2;
                            const ulonglong2 wa = *reinterpret_cast<const ulonglong2*>(dwp);
                            const ulonglong2 wb = *reinterpret_cast<const ulonglong2*>(dwp + 4);
                            csc[0] = wa.x; csc[1] = wa.y; csc[2] = wb.x; csc[3] = wb.y;
#pragma unroll
                            for (int k = 0; k < 2; ++k) {                  // 16-column halves
                                const uint32_t ta = taddr + h * BN + 16 * k;
                                uint32_t s0[8], s1[8];
                                tmem_ld16x256b_x2(ta, s0);                 // lanes rb, rb + 8
                                tmem_ld16x256b_x2(ta + (16u << 16), s1);   // lanes rb + 16, rb + 24
                                tmem_wait_ld();
                                if (h == 1 && k == 1) {                    // pair slot read out
                                    tc_fence_before();
                                    __syncwarp();
                                    if (lane == 0) mbar_arrive(B.tempty + 8 * ps);
                                }
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float d = h ? lsc[i].y : lsc[i].x;
                                    const uint64_t d2 = pack2(d, d);
                                    const uint32_t* sv = i < 2 ? s0 : s1;
                                    const int e = 2 * (i & 1);
                                    fma_f32x2(acc[i][2 * k], mul_f32x2(pack2u(sv[e], sv[e + 1]), csc[2 * k]), d2);
                                    fma_f32x2(acc[i][2 * k + 1], mul_f32x2(pack2u(sv[4 + e], sv[4 + e + 1]), csc[2 * k + 1]), d2);
                                }
                            }
                        }
                    } else {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(B.tempty + 8 * ps);
                    }
                    if ((g0 + 1) % SCG == SCG - 1) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(B.empty_sc + 8 * slot);
                        ++sc;
                    }
                }
                if (!ok) break;
                if (live) {
                    const Unit uu = unit_at(t, PAIRS, ta);                 // again: fewer live registers
                    const Tile T = tile_at<kGrouped>(uu.tile, M, G, ga, n_tiles);
                    {
                        // a tail chunk stores into its partial slot (BN columns, 8-byte aligned)
                        const bool part = uu.slot >= 0;
                        float* ybase = part ? ta.part + (int64_t)uu.slot * (BM * BN) + cb + c2
                                            : y + T.m0 * ldy + T.n0 + cb + c2;
                        const int64_t ld = part ? BN : ldy;
                        const bool v2 = vec2 || part;
                        const int64_t col0 = T.n0 + cb + c2;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int row = rb + 8 * i;                   // tile row
                            if (row < T.rows) {
                                float* yr = ybase + row * ld;
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const float2 v = unpack2(acc[i][j]);
                                    const int64_t col = col0 + 8 * j;
                                    if (v2 && col + 1 < N) {
                                        *reinterpret_cast<float2*>(yr + 8 * j) = v;
                                    } else {
                                        if (col < N) yr[8 * j] = v.x;
                                        if (col + 1 < N) yr[8 * j + 1] = v.y;
                                    }
                                }
                            }
                        }
                    }
                }
            }
          }
        }

    // this CTA's tiles are done: the next kernel on the stream may start
    // launching (it still waits for the whole grid before it reads anything)
    pdl_release();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---- pre-pass: int8 codes -> binary16 (optionally gathered) ---------------------------
//
// Each step is written as the work of block blk of nblk blocks (a grid-stride
// range), so that the dense product can run all three of its steps in one
// launch (dense_prepass_kernel) and the grouped product its gather alone.

// Dense: a16[r] = fp16(qx[r]).  Grouped (perm != nullptr): sorted position i
// takes activation row x_row(perm[i]); its scales are gathered into dxg too.
__device__ __forceinline__ void widen_rows_range(const int8_t* __restrict__ qx, const float* __restrict__ dx,
                                                 int64_t rows, int64_t K, __half* __restrict__ a16,
                                                 float* __restrict__ dxg, const int32_t* __restrict__ perm,
                                                 const int32_t* __restrict__ n_rows, int32_t topk,
                                                 int32_t x_row_mode, int64_t blk, int64_t nblk) {
    const int64_t chunks = K / 16;                   // 16 codes per thread step
    const int64_t G = K / kGroup;
    const int64_t limit = n_rows ? (int64_t)*n_rows : rows;
    const int64_t total = limit * chunks;
    for (int64_t i = blk * blockDim.x + threadIdx.x; i < total; i += nblk * blockDim.x) {
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

// Dense Q4 weights -> binary16 [N][K]: one packed 16-byte group per thread
// step (byte j: element j in the low nibble, element j + 16 in the high
// nibble, each stored q + 8), written as 64 bytes of binary16 in element order.
__device__ __forceinline__ void widen_q4_range(const uint8_t* __restrict__ qw4, int64_t groups,
                                               __half* __restrict__ w16, int64_t blk, int64_t nblk) {
    for (int64_t i = blk * blockDim.x + threadIdx.x; i < groups; i += nblk * blockDim.x) {
        const uint4 v = *reinterpret_cast<const uint4*>(qw4 + i * 16);
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
        uint4* o = reinterpret_cast<uint4*>(w16 + i * kGroup);
        o[0] = make_uint4(lo_h[0], lo_h[1], lo_h[2], lo_h[3]);
        o[1] = make_uint4(lo_h[4], lo_h[5], lo_h[6], lo_h[7]);
        o[2] = make_uint4(hi_h[0], hi_h[1], hi_h[2], hi_h[3]);
        o[3] = make_uint4(hi_h[4], hi_h[5], hi_h[6], hi_h[7]);
    }
}

// dwT[g][.]: the weight scale plane dw [N][G] (binary16) transposed to
// group-major binary32 rows of ldt columns (ldt a multiple of 32), the layout
// the epilogue reads.  Inside each 32-column block, column 8j + 2c + e is
// stored at 8c + 2j + e (j, c < 4, e < 2), so the 8 columns one epilogue
// thread scales are contiguous; columns past N are stored as zero.  One tile
// (bx, by) is 32 columns x 32 groups: dw rows are read along g into shared
// memory, then dwT rows are written along the stored column (both coalesced).
// Every thread of the block calls it (it synchronises the block).
__device__ __forceinline__ void transpose_scales_tile(const uint16_t* __restrict__ dw, int64_t N, int64_t G,
                                                      float* __restrict__ dwt, int64_t ldt, int64_t bx,
                                                      int64_t by, float (&tile)[32][33]) {
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int64_t n0 = bx * 32, g0 = by * 32;
    for (int i = ty; i < 32; i += 8) {                   // column n0 + i, group g0 + tx
        const int64_t n = n0 + i, g = g0 + tx;
        tile[i][tx] = (n < N && g < G) ? half_bits_to_float(dw[n * G + g]) : 0.f;
    }
    __syncthreads();
    // stored slot tx of the block holds column 8j + 2c + e
    const int c = tx >> 3, j = (tx >> 1) & 3, e = tx & 1;
    const int col = 8 * j + 2 * c + e;
    for (int i = ty; i < 32; i += 8) {                   // group g0 + i, stored column n0 + tx
        const int64_t g = g0 + i;
        if (g < G) dwt[g * ldt + n0 + tx] = tile[col][i];
    }
}

// The grouped product's gather (and any single widening).
__global__ void __launch_bounds__(256)
widen_rows_kernel(const int8_t* __restrict__ qx, const float* __restrict__ dx, int64_t rows,
                  int64_t K, __half* __restrict__ a16, float* __restrict__ dxg,
                  const int32_t* __restrict__ perm, const int32_t* __restrict__ n_rows,
                  int32_t topk, int32_t x_row_mode) {
    pdl_wait();                                      // the codes may come from the previous kernel
    pdl_release();
    widen_rows_range(qx, dx, rows, K, a16, dxg, perm, n_rows, topk, x_row_mode, blockIdx.x, gridDim.x);
}

// The dense product's pre-pass in one launch: blocks [0, nb_w) widen the
// weight codes, the next nb_a the activation codes, the rest transpose one
// 32 x 32 tile of the weight scales each.  The three steps touch disjoint
// buffers, so they share the HBM bandwidth instead of running one after
// another (and two launch gaps are gone).
struct DensePrepass {
    const int8_t* qx;            // activation codes [M][K]
    __half* a16;
    const void* qw;              // weight codes [N][K] (Q8) or [N][K/2] (Q4)
    __half* w16;
    const uint16_t* dw;          // weight scales [N][G]
    float* dwt;                  // [G][ldt]
    int64_t M, N, K, G, ldt;
    int nb_w, nb_a, tiles_x;     // blocks per step; scale tiles along N
    bool q4;
};

__global__ void __launch_bounds__(256)
dense_prepass_kernel(const DensePrepass a) {
    __shared__ float tile[32][33];
    pdl_wait();                                      // the codes may come from the previous kernel
    pdl_release();
    int64_t b = blockIdx.x;
    if (b < a.nb_w) {
        if (a.q4)
            widen_q4_range(static_cast<const uint8_t*>(a.qw), a.N * a.G, a.w16, b, a.nb_w);
        else
            widen_rows_range(static_cast<const int8_t*>(a.qw), nullptr, a.N, a.K, a.w16, nullptr, nullptr,
                             nullptr, 1, 0, b, a.nb_w);
        return;
    }
    b -= a.nb_w;
    if (b < a.nb_a) {
        widen_rows_range(a.qx, nullptr, a.M, a.K, a.a16, nullptr, nullptr, nullptr, 1, 0, b, a.nb_a);
        return;
    }
    b -= a.nb_a;
    transpose_scales_tile(a.dw, a.N, a.G, a.dwt, a.ldt, b % a.tiles_x, b / a.tiles_x, tile);
}

// y of the tail tiles: the sum of each tile's K-chunk partials, added in chunk
// order (deterministic).  One thread per output element of the tail tiles.
__global__ void __launch_bounds__(256)
tail_reduce_kernel(const float* __restrict__ part, int full, int split, int tail_tiles,
                   int n_tiles, int64_t M, int64_t N, float* __restrict__ y, int64_t ldy) {
    pdl_wait();                                          // the partial sums of the GEMM
    const int64_t total = (int64_t)tail_tiles * BM * BN;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int l = (int)(i / (BM * BN));
        const int r = (int)(i / BN) % BM, c = (int)(i % BN);
        const int tile = full + l;
        const int64_t m = (int64_t)(tile / n_tiles) * BM + r, n = (int64_t)(tile % n_tiles) * BN + c;
        if (m < M && n < N) {
            const float* p = part + (int64_t)l * split * (BM * BN) + r * BN + c;
            float s = p[0];
            for (int k = 1; k < split; ++k) s += p[(int64_t)k * (BM * BN)];
            y[m * ldy + n] = s;
        }
    }
}

// MoE tile table, ordered by slot width: first every tile of more than 64
// rows (full 128-row tiles and long tails), then the tails of 33-64 rows, then
// those of at most 32, each class in expert order.  A CTA walks the table with
// a stride of the grid size, so its tiles change TMEM slot layout at most
// twice per call (each change drains the pair-slot ring).  Each entry:
// {first sorted row, rows, expert, 0}; the entry count equals tile_offsets[E].
// One block of 1024 threads, experts taken 1024 at a time.
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

// Tensor maps of one product: A binary16 [rows][K], dx [rows][G] (binary32,
// row-major), and the weights: dense (ldt > 0), B binary16 [brows][K] (the
// widened codes, boxes of one pair like A's) and the scales dwT [G][ldt]
// binary32; MoE (ldt == 0), B codes [brows][K/2] and dw [brows][G] binary16 as
// stored.
bool make_maps(CUtensorMap* ma, CUtensorMap* mb, CUtensorMap* mdx, CUtensorMap* mdw,
               const void* a16, const void* qw, const float* dx, const void* dws,
               int64_t rows, int64_t brows, int64_t ldt, int64_t K, bool q4) {
    const int64_t G = K / kGroup;
    const int64_t wbytes = q4 ? K / 2 : K;
    const bool dw_ok = ldt > 0
        ? make_map(mdw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dws, ldt, G, ldt * 4, BN, SCG,
                   CU_TENSOR_MAP_SWIZZLE_NONE)
        : make_map(mdw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, dws, G, brows, G * 2, SCG, BN,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    return dw_ok &&
           make_map(mdx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dx, G, rows, G * 4, SCG, BM,
                    CU_TENSOR_MAP_SWIZZLE_NONE) &&
           make_map(ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a16, K, rows, K * 2, 64, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           (ldt > 0 ? make_map(mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qw, K, brows, K * 2, 64, BN,
                               CU_TENSOR_MAP_SWIZZLE_128B)
                    : make_map(mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, wbytes, brows, wbytes, 128, BN,
                               CU_TENSOR_MAP_SWIZZLE_128B));
}

template <bool kQ4, bool kGrouped>
cudaError_t launch_kernel(dim3 grid, const CUtensorMap& ma, const CUtensorMap& mb,
                          const CUtensorMap& mdx, const CUtensorMap& mdw, float* y, int64_t M,
                          int64_t N, int64_t K, int64_t ldy, GroupedArgs ga, int n_tiles,
                          int64_t dense_tiles, TailArgs ta, cudaStream_t s) {
    cudaError_t e = ensure_smem_attr((const void*)tc_gemm_kernel<kQ4, kGrouped>, SMEM_BYTES,
                                     9 + (kQ4 ? 1 : 0) + (kGrouped ? 2 : 0));
    if (e != cudaSuccess) return e;
    const bool vec2 = ((uintptr_t)y % 8 == 0) && (ldy % 2 == 0);
    return launch_pdl(tc_gemm_kernel<kQ4, kGrouped>, grid, dim3(kGrouped ? THREADS : THREADS_DENSE),
                      (size_t)SMEM_BYTES, s, ma, mb, mdx, mdw, y, M, N, K, ldy, vec2, ga, n_tiles,
                      dense_tiles, ta);
}

// Tail split of a dense product with `tiles` output tiles and G groups: the
// tiles of the last, partly empty round of a one-CTA-per-SM grid (all of them
// when there are fewer tiles than SMs) are cut into the most K chunks that
// still fit that round, each a multiple of 8 groups.
struct TailPlan {
    int64_t full, tail;    // whole-tile units; tail tiles
    int split;             // chunks per tail tile (1: none)
};

TailPlan tail_plan(int64_t tiles, int64_t G) {
    const int64_t sms = sm_count();
    TailPlan p{tiles, 0, 1};
    if (sms <= 0) return p;
    const int64_t L = tiles % sms;
    if (L == 0) return p;
    int64_t s = sms / L;
    while (s > 1 && (G / 8) % s != 0) --s;
    if (s > 1) {
        p.full = tiles - L;
        p.tail = L;
        p.split = (int)s;
    }
    return p;
}

size_t tail_bytes(const TailPlan& p) { return (size_t)p.tail * p.split * BM * BN * 4; }

int widen_grid(int64_t work) {
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

size_t align16(size_t v) { return (v + 15) / 16 * 16; }

}  // namespace

int tc_tile_m() { return BM; }

// TMA coordinates and the tile arithmetic are 32-bit: rows and columns below
// 2^31 - 256.
bool tc_gemm_supported(int64_t M, int64_t N, int64_t K, const void* dx, const void* dw) {
    constexpr int64_t kMax = (1ll << 31) - 256;
    return K % 256 == 0 && M < kMax && N < kMax && K < kMax &&
           ((uintptr_t)dx % 16 == 0) && ((uintptr_t)dw % 16 == 0) && encoder() != nullptr;
}

int64_t ldt_of(int64_t N) { return (N + 31) / 32 * 32; }

int64_t dense_tile_count(int64_t M, int64_t N) { return ((N + BN - 1) / BN) * ((M + BM - 1) / BM); }

// dense workspace: a16 [M][K] binary16 | dwT [G][ldt(N)] binary32 | w16 [N][K]
// binary16 (the weight codes widened) | the tail tiles' K-chunk partials
// (binary32, BM x BN each; none without a tail split)
size_t tc_gemm_workspace(int64_t M, int64_t N, int64_t K, bool q4) {
    (void)q4;
    const int64_t G = K / kGroup;
    return align16((size_t)M * K * 2) + align16((size_t)G * ldt_of(N) * 4) +
           align16((size_t)N * K * 2) + tail_bytes(tail_plan(dense_tile_count(M, N), G));
}

cudaError_t launch_tc_gemm(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                           const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                           void* workspace, cudaStream_t s) {
    const int64_t G = K / kGroup, ldt = ldt_of(N);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    __half* a16 = reinterpret_cast<__half*>(ws);
    const size_t off_dwt = align16((size_t)M * K * 2);
    const size_t off_w16 = off_dwt + align16((size_t)G * ldt * 4);
    const size_t off_part = off_w16 + align16((size_t)N * K * 2);
    float* dwt = reinterpret_cast<float*>(ws + off_dwt);
    __half* w16 = reinterpret_cast<__half*>(ws + off_w16);
    // the pre-pass and the GEMM are programmatic dependent launches: each
    // waits for its predecessor before reading, so a launch and its set-up
    // overlap the end of the kernel before it
    const int sm = sm_count();
    DensePrepass pa;
    pa.qx = qx; pa.a16 = a16; pa.qw = qw; pa.w16 = w16; pa.dw = dw; pa.dwt = dwt;
    pa.M = M; pa.N = N; pa.K = K; pa.G = G; pa.ldt = ldt; pa.q4 = q4;
    const int64_t w_items = q4 ? N * G : N * (K / 16), a_items = M * (K / 16);
    pa.nb_w = (int)min64((w_items + 255) / 256, (int64_t)sm * 4);
    pa.nb_a = (int)min64((a_items + 255) / 256, (int64_t)sm * 2);
    if (pa.nb_w < 1) pa.nb_w = 1;
    if (pa.nb_a < 1) pa.nb_a = 1;
    pa.tiles_x = (int)(ldt / 32);
    const int64_t nb_t = (int64_t)pa.tiles_x * ((G + 31) / 32);
    cudaError_t e = launch_pdl(dense_prepass_kernel, dim3((unsigned)(pa.nb_w + pa.nb_a + nb_t)), dim3(256), 0,
                               s, pa);
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb, mdx, mdw;
    if (!make_maps(&ma, &mb, &mdx, &mdw, a16, w16, dx, dwt, M, N, ldt, K, q4))
        return cudaErrorInvalidValue;
    const int n_tiles = (int)((N + BN - 1) / BN);
    const int64_t tiles = dense_tile_count(M, N);
    const TailPlan tp = tail_plan(tiles, G);
    const int64_t units = tp.full + tp.tail * tp.split;
    const int64_t ctas = units < sm_count() ? units : sm_count();
    dim3 grid((unsigned)ctas);
    GroupedArgs ga{};
    float* part = reinterpret_cast<float*>(ws + off_part);
    const TailArgs ta{(int)tp.full, tp.split, part};
    e = q4 ? launch_kernel<true, false>(grid, ma, mb, mdx, mdw, y, M, N, K, ldy, ga, n_tiles, units, ta, s)
           : launch_kernel<false, false>(grid, ma, mb, mdx, mdw, y, M, N, K, ldy, ga, n_tiles, units, ta, s);
    if (e != cudaSuccess || tp.tail == 0) return e;
    const int64_t elems = tp.tail * BM * BN;
    return launch_pdl(tail_reduce_kernel, dim3(widen_grid(elems)), dim3(256), 0, s, (const float*)part,
                      (int)tp.full, tp.split, (int)tp.tail, n_tiles, M, N, y, ldy);
}

// MoE workspace after the routing tables: a16 [P][K] binary16 and dxg [P][G]
// binary32 (gathered activation rows and scales in expert order), and the
// m-tile table (at most P / 128 + E tiles, 16 bytes each).
int4* tc_grouped_tile_table(void* workspace, int64_t P, int64_t K) {
    const int64_t G = K / kGroup;
    return reinterpret_cast<int4*>(static_cast<uint8_t*>(workspace) + align16((size_t)P * K * 2) +
                                   align16((size_t)P * G * 4));
}

size_t tc_grouped_workspace(int64_t P, int64_t N, int64_t K, int32_t E) {
    (void)N;
    const int64_t G = K / kGroup;
    return align16((size_t)P * K * 2) + align16((size_t)P * G * 4) +
           (size_t)(P / BM + E + 1) * 16;
}

cudaError_t launch_tc_grouped(const int8_t* qx, const float* dx, int64_t P, int64_t N, int64_t K,
                              const uint8_t* qw4, const uint16_t* dw, float* y, int32_t E,
                              int32_t topk, int32_t x_row_mode, const int32_t* perm,
                              const int32_t* offsets, const int32_t* tile_offsets,
                              void* workspace, cudaStream_t s) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    __half* a16 = reinterpret_cast<__half*>(ws);
    float* dxg = reinterpret_cast<float*>(ws + align16((size_t)P * K * 2));
    int4* info = tc_grouped_tile_table(workspace, P, K);      // filled by the routing kernel
    // gather + widen the routed rows (count read on the device: offsets[E])
    cudaError_t e = launch_pdl(widen_rows_kernel, dim3(widen_grid(P * (K / 16))), dim3(256), 0, s, qx, dx,
                               P, K, a16, dxg, perm, offsets + E, topk, x_row_mode);
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb, mdx, mdw;
    if (!make_maps(&ma, &mb, &mdx, &mdw, a16, qw4, dxg, dw, P, (int64_t)E * N, 0, K, true))
        return cudaErrorInvalidValue;
    const int n_tiles = (int)((N + BN - 1) / BN);
    GroupedArgs ga{perm, offsets, tile_offsets, info, E, N};
    dim3 grid((unsigned)sm_count());
    return launch_kernel<true, true>(grid, ma, mb, mdx, mdw, y, P, N, K, N, ga, n_tiles, 0,
                                     TailArgs{0, 1, nullptr}, s);
}

cudaError_t set_wait_limit(long long cycles) {
    const long long v = cycles > 0 ? cycles : kWaitCycles;
    return cudaMemcpyToSymbol(g_wait_limit, &v, sizeof v);
}

unsigned int read_and_clear_tc_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    cudaMemcpyToSymbol(g_tc_error, &z, sizeof z);
    return v;
}

}  // namespace qg
