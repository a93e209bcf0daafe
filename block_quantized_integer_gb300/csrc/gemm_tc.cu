// Prefill GEMM and grouped MoE GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA).
//
// y[m,n] = sum_g dw[n,g] dx[m,g] S[m,n,g] with S the exact integer dot
// product of one 32-group ("I wrote a custom CUDA inference engine to run
// Qwen3.5-27B on a $130 mining card", Features: the Q8_0 GEMM tile path of the
// prefill; "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU",
// Methodology 1: grouped 4-bit GEMM for MoE routing; Methodology 2: 4-bit
// weights with 8-bit activations; Methodology 4: one pass over the whole
// prompt keeps the GEMM M large).
//
// sm_103a has no integer tcgen05 MMA form, so the codes are widened to
// binary16, where every value in [-127, 127] is exact, and multiplied with
// kind::f16 into binary32 tensor memory: each product is an integer below
// 2^14 and each group sum an integer below 2^19, which the tensor core
// accumulates without loss (the group-dot tests check this bit for bit).
//
// Tile: 128 TMEM lanes (activation rows) x 256 weight rows (the MMA's N), K
// walked one group at a time.  Each group's S goes to one of two 256-column
// TMEM slots (two K=16 MMAs, the first overwrites), so the MMAs of group g+1
// run while the epilogue reads group g.  An MMA of N = 256 keeps the tensor
// pipe busy for ~128 cycles, long enough to hide the issuing thread's barrier
// probes and commits; at N = 128 they were not hidden (measured).
//
// Two kernel forms:
//  plain (dense Q8_0; 640 threads): activation and weight codes widened to
//    binary16 by a pre-pass, weight scales transposed to binary32 [G][cols]
//    (the layout the epilogue reads) by a pre-pass; 128-row m-tiles.
//  conv (dense Q4_0 and the grouped MoE product; 768 threads): 4 converter
//    warps unpack the 4-bit weight codes in shared memory into the binary16
//    operand (no widened copy of the weights in HBM) and transpose each
//    stage of binary16 weight scales; 64-row m-tiles, whose rows are spread
//    over the four TMEM lane quarters (c = ceil(rows / 4) rows each, loaded
//    as four TMA boxes) so that all four SM sub-partitions share the epilogue
//    even for a short MoE segment.
//
// Warp roles (persistent: one CTA per SM walks work items b, b + grid, ...):
//   warps 0-15  epilogue: warp w reads lane quarter w % 4, columns
//               64 (w / 4) .. +63, as 16-lane x 256-bit fragments, releases
//               the TMEM slot once read, and adds (S * dw) * dx on packed
//               f32x2 instructions into binary32 registers; y is written once
//               per work item.
//   warp 16     TMA producer: binary16 A (one pair of groups, 128-byte
//               swizzle), plain: binary16 B of the pair; conv: packed 4-bit B
//               (4 groups, 64-byte swizzle); scale stages every 8 groups.
//   warp 17     MMA issuer (one thread): per group two K=16 MMAs into a TMEM
//               slot and a commit; per pair a commit that frees the operand
//               slot.
//   warps 18-19 idle (their registers go to the epilogue warps).
//   warps 20-23 (conv) converters: two B rows per thread, 4-bit codes ->
//               binary16 into the operand slot in the 128-byte-swizzled layout
//               the MMA reads; binary16 weight scales -> binary32 [g][col].
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

namespace {

using namespace tc;

constexpr int BM = 128;                // MMA M: TMEM lanes
constexpr int BN = 256;                // MMA N: weight rows of a tile
constexpr int NSLOT = 2;               // TMEM group slots of BN columns
constexpr int SCG = 8;                 // groups per scale stage
constexpr int EPI_WARPS = 16;          // 4 per TMEM lane quarter, 64 columns each
// Warpgroups: 0-3 epilogue, 4 producer (warp 16) + MMA issuer (warp 17) + two
// idle warps, 5 (conv form) converters.  Roles follow warpgroup lines so that
// setmaxnreg can move registers from the light roles to the epilogue.
constexpr int PROD_WARP = 16, MMA_WARP = 17, CONV_WARP0 = 20, CONV_WARPS = 4;
constexpr int CONV_THREADS = CONV_WARPS * 32;              // 128: two B rows each
constexpr int THREADS_PLAIN = 20 * 32;                     // 640
constexpr int THREADS_CONV = THREADS_PLAIN + CONV_THREADS;  // 768

constexpr int A_SLOT = BM * 128;       // 16 KiB: 128 rows x one pair of groups, binary16
constexpr int B_SLOT = BN * 128;       // 32 KiB: 256 rows x one pair of groups, binary16
constexpr int OP_SLOT = A_SLOT + B_SLOT;
constexpr int QB_STAGE = BN * 64;      // 16 KiB: 256 rows x 4 groups of packed 4-bit codes
constexpr int SC_DX = BM * SCG * 4;    // dx [128 lanes][8 groups] binary32
constexpr int SC_DWT = SCG * BN * 4;   // dw [8 groups][256 columns, permuted] binary32
constexpr int SC_DWRAW = BN * SCG * 2; // conv: dw as stored, [256 rows][8 groups] binary16

template <bool kConv>
struct Cfg {
    static constexpr int THREADS = kConv ? THREADS_CONV : THREADS_PLAIN;
    // Registers a thread: the launch gives every thread LAUNCH_REGS (the
    // compiler's bound for THREADS threads); the warpgroups then trade them,
    // and their shares add up to exactly the launch's THREADS x LAUNCH_REGS.
    static constexpr int LAUNCH_REGS = kConv ? 80 : 96;
    static constexpr int EPI_REGS = kConv ? 96 : 112;
    static constexpr int CTRL_REGS = kConv ? 32 : 24;       // producer, MMA issuer, idle
    static constexpr int CONV_REGS = 64;
    static_assert(4 * 128 * EPI_REGS + 128 * CTRL_REGS + (kConv ? 128 * CONV_REGS : 0) <=
                  THREADS * LAUNCH_REGS, "register shares must add up to the launch's registers");
    static constexpr int ROWS = kConv ? 64 : 128;           // activation rows of an m-tile
    static constexpr int QROWS = ROWS / 4;                  // rows per lane quarter (full tile)
    static constexpr int NO = kConv ? 3 : 4;                // operand slots
    static constexpr int NB = kConv ? 2 : 0;                // packed 4-bit B stages
    static constexpr int NSC = 2;                           // scale stages
    static constexpr int SC_STAGE = SC_DX + SC_DWT + (kConv ? SC_DWRAW : 0);
    static constexpr int OFF_OP = 0;
    static constexpr int OFF_QB = OFF_OP + NO * OP_SLOT;
    static constexpr int OFF_SC = OFF_QB + NB * QB_STAGE;
    static constexpr int OFF_BAR = OFF_SC + NSC * SC_STAGE;
    static constexpr int NUM_BARS = 2 * NO + 2 * NSLOT + 3 * NSC + 2 * NB + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;       // + alignment slack
    // A bytes of one pair: plain one 128-row box, conv four boxes of QROWS rows
    static constexpr uint32_t A_BYTES = kConv ? 4 * QROWS * 128 : BM * 128;
    static constexpr uint32_t DX_BYTES = kConv ? 4 * QROWS * SCG * 4 : SC_DX;
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(OFF_QB % 1024 == 0 && OFF_SC % 1024 == 0 && SC_STAGE % 1024 == 0,
                  "swizzled stages need 1 KiB alignment");
};

constexpr uint32_t TMEM_COLS = NSLOT * BN;           // 512
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
constexpr uint32_t kSpinLimit = 1u << 22;            // drain polls after an abort
constexpr long long kWaitCycles = 4000000000ll;      // ~2 s at 2 GHz: a wait that long has failed
constexpr uint32_t kSleepHintNs = 20000;             // a waiter sleeps until the phase flips

// full: the operand slot holds both operands of a pair (TMA bytes landed; conv:
// and the converters wrote the binary16 B); done: the pair's MMAs completed
// (slot free); afull: a TMEM slot's MMAs completed; tempty: the epilogue read
// the TMEM slot; full_sc: a scale stage is ready for the epilogue (conv: after
// the converters transposed dw); empty_sc: the epilogue is done with it;
// full_raw (conv): the scale stage's TMA bytes landed; full_b / empty_b (conv):
// packed 4-bit B stages.
struct Bars {
    uint32_t full, done, afull, tempty, full_sc, empty_sc, full_raw, full_b, empty_b, drain;
};

template <bool kConv>
__device__ __forceinline__ Bars bars_at(uint32_t base) {
    using C = Cfg<kConv>;
    Bars b;
    b.full = base;
    b.done = b.full + 8 * C::NO;
    b.afull = b.done + 8 * C::NO;
    b.tempty = b.afull + 8 * NSLOT;
    b.full_sc = b.tempty + 8 * NSLOT;
    b.empty_sc = b.full_sc + 8 * C::NSC;
    b.full_raw = b.empty_sc + 8 * C::NSC;
    b.full_b = b.full_raw + 8 * C::NSC;
    b.empty_b = b.full_b + 8 * C::NB;
    b.drain = b.empty_b + 8 * C::NB;
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

// Register reallocation of the calling warpgroup (all its warps execute it).
template <int R>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(R));
}
template <int R>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(R));
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
// One packed 16-byte Q4 group (byte j: element j in the low nibble, element
// j + 16 in the high nibble) -> its 32 binary16 values as four 16-byte chunks
// in element order.
__device__ __forceinline__ void q4_group_to_h32(const uint4 v, uint4 (&o)[4]) {
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
    o[0] = make_uint4(lo_h[0], lo_h[1], lo_h[2], lo_h[3]);
    o[1] = make_uint4(lo_h[4], lo_h[5], lo_h[6], lo_h[7]);
    o[2] = make_uint4(hi_h[0], hi_h[1], hi_h[2], hi_h[3]);
    o[3] = make_uint4(hi_h[4], hi_h[5], hi_h[6], hi_h[7]);
}

// Column permutation of the binary32 weight-scale rows [g][256]: inside each
// 64-column span (one epilogue warp's columns), column 16k + 8j + 2c + e is
// stored at 16c + 4k + 2j + e (k, c < 4; j, e < 2), so the 16 columns one
// epilogue thread scales are contiguous (four 16-byte loads a group).
__host__ __device__ __forceinline__ int dw_perm(int col) {
    const int s = col & ~63, x = col & 63;
    const int k = x >> 4, j = (x >> 3) & 1, c = (x >> 1) & 3, e = x & 1;
    return s + 16 * c + 4 * k + 2 * j + e;
}

struct GroupedArgs {
    const int32_t* perm;          // sorted position -> pair index
    const int32_t* tile_offsets;  // [E+1] in m-tiles; tile_offsets[E] = m-tile count
    const int4* tile_info;        // per m-tile: {first sorted row, rows, expert, 0}
    int32_t E;
    int64_t N;                    // per-expert output columns
};

// Dense work units.  Units [0, full) are whole output tiles.  When the tile
// count leaves the last round of the persistent grid partly empty, each of
// those last tiles is cut along K into `split` chunks of equal length (a
// multiple of 8 groups, so every stage boundary stays where it was): unit
// full + l * split + c is chunk c of tile full + l.  A chunk's binary32 sums go
// to partial slot l * split + c of `part` (BM x BN each, rows in lane order),
// and tail_reduce_kernel adds a tile's chunks in chunk order into y.
struct TailArgs {
    int full;          // whole-tile units
    int split;         // K chunks per tail tile (1: no tail split)
    float* part;       // [(units - full)][BM][BN] binary32
};

// One work item: an m-tile of activation rows x a tile of BN weight rows,
// over groups [g0, g0 + ng).  Lane l of quarter q holds activation row
// m0 + q * c + l (valid when l < c and q * c + l < rows).
struct Item {
    int m0;           // first activation row (dense) / sorted row (MoE)
    int n0;           // first output column
    int bn0;          // first weight row in the B plane
    int rows, c;      // valid rows; rows per lane quarter
    int g0, ng;       // group range
    int slot;         // tail partial slot (-1: y)
};

template <bool kConv, bool kGrouped>
__device__ __forceinline__ Item item_at(int t, int64_t M, int G, int n_tiles, const GroupedArgs& ga,
                                        const TailArgs& ta) {
    using C = Cfg<kConv>;
    Item it;
    int tile = t;
    it.g0 = 0;
    it.ng = G;
    it.slot = -1;
    if constexpr (!kGrouped) {
        if (t >= ta.full) {
            const int v = t - ta.full;
            it.ng = G / ta.split;
            tile = ta.full + v / ta.split;
            it.g0 = it.ng * (v % ta.split);
            it.slot = v;
        }
    }
    const int mt = tile / n_tiles;
    it.n0 = (tile % n_tiles) * BN;
    if constexpr (kGrouped) {
        const int4 info = ga.tile_info[mt];
        it.m0 = info.x;
        it.rows = info.y;
        it.c = (info.y + 3) >> 2;
        it.bn0 = info.z * (int)ga.N + it.n0;
    } else {
        it.m0 = mt * C::ROWS;
        it.rows = (int)min64(C::ROWS, M - it.m0);
        it.c = C::QROWS;
        it.bn0 = it.n0;
    }
    return it;
}

// Epilogue of one work item.  NI: 8-lane slots of its quarter a thread uses
// (lanes q * 32 + lane / 4 + 8 i, i < NI): 1 or 2 when c <= 8 or 16, 4 for
// 128-row tiles.  Per group: wait for the TMEM slot, read it in four 16-column
// chunks (16x256b fragments: lane slot i, block j holds columns
// 16k + 8j + 2 (lane % 4) + {0, 1}), release the slot after the last read,
// and add (S * dw) * dx into acc.  Each output is one thread's running sum
// over the groups in order.  Returns false when a wait gave up.
template <bool kConv, bool kGrouped, int NI>
__device__ __forceinline__ bool epilogue_item(uint32_t bars, const uint8_t* smem, uint32_t tmem_base,
                                              volatile int* abort, int t, int64_t M, int G, int n_tiles,
                                              const GroupedArgs& ga, const TailArgs& ta, uint32_t& gc,
                                              uint32_t& sc, int warp, int lane,
                                              float* __restrict__ y, int64_t N, int64_t ldy, bool vec2) {
    using C = Cfg<kConv>;
    const int q = warp & 3, cw = warp >> 2;
    const int tq = lane >> 2, c4 = lane & 3;
    int g0, ng;
    bool live;
    {
        const Item it = item_at<kConv, kGrouped>(t, M, G, n_tiles, ga, ta);
        g0 = it.g0;
        ng = it.ng;
        // a warp whose quarter holds no valid row keeps the barrier protocol
        // but skips the readout and math
        live = q * it.c < it.rows;
    }
    uint64_t acc[NI][8];
#pragma unroll
    for (int i = 0; i < NI; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0ull;
    for (int gi = 0; gi < ng; ++gi, ++gc) {
        const Bars B = bars_at<kConv>(bars);
        const int g = g0 + gi;
        const int ts = (int)(gc & 1);
        const int sslot = (int)(sc % C::NSC);
        if (g % SCG == 0 && !wait_bar<true>(B.full_sc + 8 * sslot, (sc / C::NSC) & 1, abort)) return false;
        if (!wait_bar<true>(B.afull + 8 * ts, (gc >> 1) & 1, abort)) return false;
        tc_fence_after();
        if (live) {
            const uint8_t* st = smem + C::OFF_SC + sslot * C::SC_STAGE;
            const float* dxs = reinterpret_cast<const float*>(st);
            const float* dws = reinterpret_cast<const float*>(st + SC_DX) + (g % SCG) * BN + cw * 64 + 16 * c4;
            float dxv[NI];
#pragma unroll
            for (int i = 0; i < NI; ++i) dxv[i] = dxs[(q * 32 + tq + 8 * i) * SCG + (g % SCG)];
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ts * BN + cw * 64);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t s0[8], s1[8];
                tmem_ld16x256b_x2(taddr + 16 * k, s0);                      // lanes tq, tq + 8
                if constexpr (NI == 4) tmem_ld16x256b_x2(taddr + 16 * k + (16u << 16), s1);
                tmem_wait_ld();
                if (k == 3) {                                               // slot read out
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B.tempty + 8 * ts);
                }
                const ulonglong2 w = *reinterpret_cast<const ulonglong2*>(dws + 4 * k);
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    const uint32_t* sv = i < 2 ? s0 : s1;
                    const int e = 2 * (i & 1);
                    const uint64_t d2 = pack2(dxv[i], dxv[i]);
                    fma_f32x2(acc[i][2 * k], mul_f32x2(pack2u(sv[e], sv[e + 1]), w.x), d2);
                    fma_f32x2(acc[i][2 * k + 1], mul_f32x2(pack2u(sv[4 + e], sv[4 + e + 1]), w.y), d2);
                }
            }
        } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.tempty + 8 * ts);
        }
        if (g % SCG == SCG - 1) {
            __syncwarp();
            if (lane == 0) mbar_arrive(B.empty_sc + 8 * sslot);
            ++sc;
        }
    }
    if (!live) return true;
    const Item it = item_at<kConv, kGrouped>(t, M, G, n_tiles, ga, ta);   // again: fewer live registers
    // columns of acc[i][2k + j]: 16k + 8j + 2 c4 + {0, 1} of the warp's 64
    const int colw = cw * 64 + 2 * c4;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int l = tq + 8 * i;
        if (l >= it.c || q * it.c + l >= it.rows) continue;
        float* yr;
        int64_t col0;
        bool v2 = vec2;
        if constexpr (kGrouped) {
            yr = y + (int64_t)ga.perm[it.m0 + q * it.c + l] * ldy;
            col0 = it.n0 + colw;
        } else if (it.slot >= 0) {
            yr = ta.part + (int64_t)it.slot * (BM * BN) + (int64_t)(q * 32 + l) * BN - it.n0;
            col0 = it.n0 + colw;
            v2 = true;
        } else {
            yr = y + (int64_t)(it.m0 + q * it.c + l) * ldy;
            col0 = it.n0 + colw;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int64_t col = col0 + 16 * k + 8 * j;
                const float2 v = unpack2(acc[i][2 * k + j]);
                if (v2 && col + 1 < N) {
                    *reinterpret_cast<float2*>(yr + col) = v;
                } else {
                    if (col < N) yr[col] = v.x;
                    if (col + 1 < N) yr[col + 1] = v.y;
                }
            }
    }
    return true;
}

// Converters (conv form): for pair p of the item, groups (g0, g0 + 1) of the
// packed stage -> binary16 B in the operand slot, 128-byte swizzled K-major
// (row r, 16-byte chunk x at r * 128 + ((x ^ (r % 8)) * 16)); the packed stage
// is 64-byte swizzled (row r, group chunk x at r * 64 + ((x ^ (r / 2 % 4)) * 16)).
// Thread ct owns B rows ct and ct + 128; all shared loads go out before any store.
__device__ __forceinline__ void convert_pair(const uint8_t* qb, uint8_t* b16, int gi, int ct) {
    uint4 v[2][2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = ct + 128 * rr;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            v[rr][h] = *reinterpret_cast<const uint4*>(qb + r * 64 + ((((gi + h) ^ (r >> 1)) & 3) << 4));
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = ct + 128 * rr;
        uint8_t* row = b16 + r * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 o[4];
            q4_group_to_h32(v[rr][h], o);
#pragma unroll
            for (int x = 0; x < 4; ++x)
                *reinterpret_cast<uint4*>(row + (((4 * h + x) ^ (r & 7)) << 4)) = o[x];
        }
    }
}

// Converters: the raw binary16 scale stage [256 rows][8 groups] -> binary32
// [8 groups][256 columns, dw_perm order].  Thread ct owns rows ct and ct + 128.
__device__ __forceinline__ void convert_scales(const uint8_t* raw, float* dwt, int ct) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = ct + 128 * rr;
        const uint4 v = *reinterpret_cast<const uint4*>(raw + r * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const int pc = dw_perm(r);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[t]));
            dwt[(2 * t) * BN + pc] = f.x;
            dwt[(2 * t + 1) * BN + pc] = f.y;
        }
    }
}

// Persistent: CTA b takes work items b, b + gridDim.x, ...  All roles walk the
// same item sequence; ring positions and barrier phases run on across items.
template <bool kConv, bool kGrouped>
__global__ void __launch_bounds__(Cfg<kConv>::THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_dx, const __grid_constant__ CUtensorMap map_dw,
               float* __restrict__ y, int64_t M, int64_t N, int64_t K, int64_t ldy, bool vec2,
               GroupedArgs ga, int n_tiles, int dense_units, TailArgs ta) {
    using C = Cfg<kConv>;
    static_assert(kConv || !kGrouped, "the grouped product has 4-bit weights");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Bars B = bars_at<kConv>(sbase + C::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const int G = (int)(K / kGroup);                    // multiple of 8
    const int num_items = kGrouped ? ga.tile_offsets[ga.E] * n_tiles : dense_units;
    const int t0 = blockIdx.x, dt = gridDim.x;

    if (tid == 0) {
        for (int i = 0; i < C::NO; ++i) {
            mbar_init(B.full + 8 * i, kConv ? 1 + CONV_WARPS : 1);
            mbar_init(B.done + 8 * i, 1);
        }
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(B.afull + 8 * i, 1);
            mbar_init(B.tempty + 8 * i, EPI_WARPS);
        }
        for (int i = 0; i < C::NSC; ++i) {
            mbar_init(B.full_sc + 8 * i, kConv ? CONV_WARPS : 1);
            mbar_init(B.empty_sc + 8 * i, EPI_WARPS);
            mbar_init(B.full_raw + 8 * i, 1);
        }
        for (int i = 0; i < C::NB; ++i) {
            mbar_init(B.full_b + 8 * i, 1);
            mbar_init(B.empty_b + 8 * i, CONV_WARPS);
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

    // each role's register share is set at the top of its own branch
    if (warp >= EPI_WARPS && warp < CONV_WARP0) {
      reg_dealloc<C::CTRL_REGS>();
      if (warp == PROD_WARP) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t ia = 0, ib = 0, isc = 0;     // stages issued so far (run on across items)
            bool ok = true;
            for (int t = t0; t < num_items && ok; t += dt) {
                const Item it = item_at<kConv, kGrouped>(t, M, G, n_tiles, ga, ta);
                // issue in the order the stages are first needed
                for (int g = it.g0; g < it.g0 + it.ng && ok; ++g) {
                    if (g % SCG == 0) {
                        const int slot = (int)(isc % C::NSC);
                        if (!(ok = wait_bar<false>(B.empty_sc + 8 * slot, ((isc / C::NSC) & 1) ^ 1, abort))) break;
                        const uint32_t dst = sbase + C::OFF_SC + slot * C::SC_STAGE;
                        const uint32_t bar = kConv ? B.full_raw + 8 * slot : B.full_sc + 8 * slot;
                        mbar_expect_tx(bar, C::DX_BYTES + (kConv ? SC_DWRAW : SC_DWT));
                        // dx row-major [rows][G] binary32: x = g, a multiple of 8 groups (32 bytes)
                        if constexpr (kConv) {
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq)
                                tma_load_2d(dst + qq * 32 * SCG * 4, &map_dx, g, it.m0 + qq * it.c, bar);
                            // dw binary16 [rows][G] as stored: x = g (16 bytes)
                            tma_load_2d(dst + SC_DX + SC_DWT, &map_dw, g, it.bn0, bar);
                        } else {
                            tma_load_2d(dst, &map_dx, g, it.m0, bar);
                            // dwT binary32 [G][ldt], permuted columns: x = n0 (1 KiB multiple)
                            tma_load_2d(dst + SC_DX, &map_dw, it.n0, g, bar);
                        }
                        ++isc;
                    }
                    if (kConv && g % 4 == 0) {
                        constexpr int NB = C::NB > 0 ? C::NB : 1;
                        const int slot = (int)(ib % NB);
                        if (!(ok = wait_bar<false>(B.empty_b + 8 * slot, ((ib / NB) & 1) ^ 1, abort))) break;
                        mbar_expect_tx(B.full_b + 8 * slot, QB_STAGE);
                        // packed 4-bit [rows][K/2]: x = 16 g bytes (64-byte multiple)
                        tma_load_2d(sbase + C::OFF_QB + slot * QB_STAGE, &map_b, g * 16, it.bn0,
                                    B.full_b + 8 * slot);
                        ++ib;
                    }
                    if (g % 2 == 0) {
                        const int slot = (int)(ia % C::NO);
                        if (!(ok = wait_bar<false>(B.done + 8 * slot, ((ia / C::NO) & 1) ^ 1, abort))) break;
                        const uint32_t op = sbase + C::OFF_OP + slot * OP_SLOT;
                        mbar_expect_tx(B.full + 8 * slot, C::A_BYTES + (kConv ? 0u : (uint32_t)B_SLOT));
                        // binary16 A [rows][K]: x = 32 g elements (64-byte multiple)
                        if constexpr (kConv) {
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq)
                                tma_load_2d(op + qq * 32 * 128, &map_a, g * 32, it.m0 + qq * it.c,
                                            B.full + 8 * slot);
                        } else {
                            tma_load_2d(op, &map_a, g * 32, it.m0, B.full + 8 * slot);
                            tma_load_2d(op + A_SLOT, &map_b, g * 32, it.bn0, B.full + 8 * slot);
                        }
                        ++ia;
                    }
                }
            }
            if (!ok) {
                for (int64_t s = (int64_t)ia - C::NO; s < (int64_t)ia; ++s)
                    if (s >= 0) drain_wait(B.full + 8 * (s % C::NO), (s / C::NO) & 1);
                if constexpr (kConv)
                    for (int64_t s = (int64_t)ib - C::NB; s < (int64_t)ib; ++s)
                        if (s >= 0) drain_wait(B.full_b + 8 * (s % C::NB), (s / C::NB) & 1);
                for (int64_t s = (int64_t)isc - C::NSC; s < (int64_t)isc; ++s)
                    if (s >= 0) drain_wait((kConv ? B.full_raw : B.full_sc) + 8 * (s % C::NSC), (s / C::NSC) & 1);
            }
        }
      } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool issued_any = false, ok = true;
            uint32_t p = 0, gc = 0;                 // pairs and groups so far
            for (int t = t0; t < num_items && ok; t += dt) {
                const int ng = item_at<kConv, kGrouped>(t, M, G, n_tiles, ga, ta).ng;
                for (int pl = 0; pl < ng / 2 && ok; ++pl, ++p) {
                    const int so = (int)(p % C::NO);
                    if (!(ok = wait_bar<false>(B.full + 8 * so, (p / C::NO) & 1, abort))) break;
                    const uint32_t a_s = sbase + C::OFF_OP + so * OP_SLOT;
                    const uint32_t b_s = a_s + A_SLOT;
#pragma unroll
                    for (int h = 0; h < 2; ++h, ++gc) {
                        const int ts = (int)(gc & 1);
                        if (!(ok = wait_bar<false>(B.tempty + 8 * ts, ((gc >> 1) & 1) ^ 1, abort))) break;
                        tc_fence_after();
                        const uint32_t d = tmem_base + (uint32_t)(ts * BN);
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            mma_f16(d, smem_desc_sw128(a_s + h * 64 + j * 32),
                                    smem_desc_sw128(b_s + h * 64 + j * 32), IDESC, j);
                        mma_commit(B.afull + 8 * ts);
                        issued_any = true;
                    }
                    if (!ok) break;
                    mma_commit(B.done + 8 * so);
                }
            }
            if (*abort && issued_any) {
                mma_commit(B.drain);
                drain_wait(B.drain, 0);
            }
        }
      }
      // warps 18 and 19 idle: their registers went to the epilogue
    } else if (warp >= CONV_WARP0) {
      // -------------------------------------------------------------- converters
      // (conv form only: the plain kernel is launched without these warps)
      reg_dealloc<C::CONV_REGS>();
      if constexpr (kConv) {
        const int ct = tid - CONV_WARP0 * 32;
        uint32_t p = 0, sb = 0, sc = 0;                     // run on across items
        bool ok = true;
        for (int t = t0; t < num_items && ok; t += dt) {
            const Item it = item_at<kConv, kGrouped>(t, M, G, n_tiles, ga, ta);
            for (int pl = 0; pl < it.ng / 2 && ok; ++pl, ++p) {
                const int g = it.g0 + 2 * pl;
                if (g % SCG == 0) {
                    const int slot = (int)(sc % C::NSC);
                    if (!(ok = wait_bar<true>(B.full_raw + 8 * slot, (sc / C::NSC) & 1, abort))) break;
                    uint8_t* st = smem + C::OFF_SC + slot * C::SC_STAGE;
                    convert_scales(st + SC_DX + SC_DWT, reinterpret_cast<float*>(st + SC_DX), ct);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B.full_sc + 8 * slot);
                    ++sc;
                }
                const int bs = (int)(sb % C::NB);
                if (g % 4 == 0 && !(ok = wait_bar<true>(B.full_b + 8 * bs, (sb / C::NB) & 1, abort))) break;
                // the operand slot is free once the MMAs of pair p - NO completed
                const int so = (int)(p % C::NO);
                if (!(ok = wait_bar<true>(B.done + 8 * so, ((p / C::NO) & 1) ^ 1, abort))) break;
                convert_pair(smem + C::OFF_QB + bs * QB_STAGE,
                             smem + C::OFF_OP + so * OP_SLOT + A_SLOT, g % 4, ct);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(B.full + 8 * so);
                    if (g % 4 == 2) mbar_arrive(B.empty_b + 8 * bs);
                }
                if (g % 4 == 2) ++sb;
            }
        }
      }
    } else {
        // ------------------------------------------------------------ epilogue
        reg_alloc<C::EPI_REGS>();
        uint32_t gc = 0, sc = 0;
        const uint32_t bars = sbase + C::OFF_BAR;
        for (int t = t0; t < num_items; t += dt) {
            bool ok;
            if constexpr (kConv) {
                const int c = item_at<kConv, kGrouped>(t, M, G, n_tiles, ga, ta).c;
                if (c <= 8)
                    ok = epilogue_item<kConv, kGrouped, 1>(bars, smem, tmem_base, abort, t, M, G, n_tiles, ga,
                                                           ta, gc, sc, warp, lane, y, N, ldy, vec2);
                else
                    ok = epilogue_item<kConv, kGrouped, 2>(bars, smem, tmem_base, abort, t, M, G, n_tiles, ga,
                                                           ta, gc, sc, warp, lane, y, N, ldy, vec2);
            } else {
                ok = epilogue_item<kConv, kGrouped, 4>(bars, smem, tmem_base, abort, t, M, G, n_tiles, ga,
                                                       ta, gc, sc, warp, lane, y, N, ldy, vec2);
            }
            if (!ok) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---- pre-passes -----------------------------------------------------------------------

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

// dwT[g][.]: the weight scale plane dw [N][G] (binary16) transposed to
// group-major binary32 rows of ldt columns (ldt a multiple of 256) in dw_perm
// order; columns past N are stored as zero.  A block takes 64 columns x 32
// groups: dw rows are read along g into shared memory, then dwT rows are
// written along the stored column (both coalesced).
__global__ void __launch_bounds__(256)
transpose_scales_kernel(const uint16_t* __restrict__ dw, int64_t N, int64_t G,
                        float* __restrict__ dwt, int64_t ldt) {
    __shared__ float tile[64][33];                       // [column][group], padded
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int64_t n0 = (int64_t)blockIdx.x * 64, g0 = (int64_t)blockIdx.y * 32;
    for (int i = ty; i < 64; i += 8) {                   // column n0 + i, group g0 + tx
        const int64_t n = n0 + i, g = g0 + tx;
        tile[i][tx] = (n < N && g < G) ? half_bits_to_float(dw[n * G + g]) : 0.f;
    }
    __syncthreads();
    // stored position s of the span holds column x with dw_perm(x) = s
    for (int i = ty; i < 32; i += 8) {                   // group g0 + i
        const int64_t g = g0 + i;
        if (g >= G) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int s = tx + 32 * h;
            const int c = s >> 4, k = (s >> 2) & 3, j = (s >> 1) & 1, e = s & 1;
            const int col = 16 * k + 8 * j + 2 * c + e;
            dwt[g * ldt + n0 + s] = tile[col][i];
        }
    }
}

// y of the tail tiles: the sum of each tile's K-chunk partials, added in chunk
// order (deterministic).  Partial row r (lane order) is activation row
// m0 + (r / 32) * qrows + r % 32 when r % 32 < qrows.  One thread per element.
__global__ void __launch_bounds__(256)
tail_reduce_kernel(const float* __restrict__ part, int full, int split, int tail_tiles,
                   int n_tiles, int rows_per_tile, int64_t M, int64_t N, float* __restrict__ y,
                   int64_t ldy) {
    const int qrows = rows_per_tile / 4;
    const int64_t total = (int64_t)tail_tiles * BM * BN;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int l = (int)(i / (BM * BN));
        const int r = (int)(i / BN) % BM, c = (int)(i % BN);
        if (r % 32 >= qrows) continue;
        const int tile = full + l;
        const int64_t m = (int64_t)(tile / n_tiles) * rows_per_tile + (r / 32) * qrows + r % 32;
        const int64_t n = (int64_t)(tile % n_tiles) * BN + c;
        if (m < M && n < N) {
            const float* p = part + (int64_t)l * split * (BM * BN) + r * BN + c;
            float s = p[0];
            for (int k = 1; k < split; ++k) s += p[(int64_t)k * (BM * BN)];
            y[m * ldy + n] = s;
        }
    }
}

// MoE m-tile table: expert e's routed rows (sorted positions offsets[e] ..
// offsets[e+1]) cut into m-tiles of at most `rows` rows, placed at
// tile_offsets[e] (the routing's exclusive scan of ceil(count / rows)).  Each
// entry: {first sorted row, rows, expert, 0}.  One thread per expert.
__global__ void __launch_bounds__(256)
tile_info_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_offsets,
                 int32_t E, int rows, int4* __restrict__ info) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const int32_t first = offsets[e], end = offsets[e + 1];
    int32_t at = tile_offsets[e];
    for (int32_t m0 = first; m0 < end; m0 += rows) info[at++] = make_int4(m0, min(rows, end - m0), e, 0);
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

// Tensor maps of one product.  A: binary16 [rows][K] (box: one pair of groups
// x 128 rows, or x 16 rows for the conv form's quarter loads); dx: binary32
// [rows][G] (8 groups x the same rows).  Plain: B binary16 [brows][K] (one
// pair x 256 rows) and dwT binary32 [G][ldt] (256 columns x 8 groups).  Conv:
// B packed 4-bit [brows][K/2] (4 groups x 256 rows, 64-byte swizzle) and dw
// binary16 [brows][G] as stored (8 groups x 256 rows).
template <bool kConv>
bool make_maps(CUtensorMap* ma, CUtensorMap* mb, CUtensorMap* mdx, CUtensorMap* mdw,
               const void* a16, const void* b, const float* dx, const void* dws,
               int64_t rows, int64_t brows, int64_t ldt, int64_t K) {
    using C = Cfg<kConv>;
    const int64_t G = K / kGroup;
    const uint32_t arows = kConv ? C::QROWS : BM;
    const bool ab = make_map(ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a16, K, rows, K * 2, 64, arows,
                             CU_TENSOR_MAP_SWIZZLE_128B) &&
                    make_map(mdx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dx, G, rows, G * 4, SCG, arows,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ab) return false;
    if constexpr (kConv)
        return make_map(mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, K / 2, brows, K / 2, 64, BN,
                        CU_TENSOR_MAP_SWIZZLE_64B) &&
               make_map(mdw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, dws, G, brows, G * 2, SCG, BN,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    else
        return make_map(mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, b, K, brows, K * 2, 64, BN,
                        CU_TENSOR_MAP_SWIZZLE_128B) &&
               make_map(mdw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dws, ldt, G, ldt * 4, BN, SCG,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <bool kConv, bool kGrouped>
cudaError_t launch_kernel(int ctas, const CUtensorMap& ma, const CUtensorMap& mb,
                          const CUtensorMap& mdx, const CUtensorMap& mdw, float* y, int64_t M,
                          int64_t N, int64_t K, int64_t ldy, GroupedArgs ga, int n_tiles,
                          int dense_units, TailArgs ta, cudaStream_t s) {
    using C = Cfg<kConv>;
    cudaError_t e = ensure_smem_attr((const void*)tc_gemm_kernel<kConv, kGrouped>, C::SMEM,
                                     9 + (kConv ? 1 : 0) + (kGrouped ? 2 : 0));
    if (e != cudaSuccess) return e;
    const bool vec2 = ((uintptr_t)y % 8 == 0) && (ldy % 2 == 0);
    tc_gemm_kernel<kConv, kGrouped><<<ctas, C::THREADS, C::SMEM, s>>>(
        ma, mb, mdx, mdw, y, M, N, K, ldy, vec2, ga, n_tiles, dense_units, ta);
    return cudaGetLastError();
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

int64_t ldt_of(int64_t N) { return (N + BN - 1) / BN * BN; }

int rows_per_tile(bool q4) { return q4 ? Cfg<true>::ROWS : Cfg<false>::ROWS; }

int64_t dense_tile_count(int64_t M, int64_t N, bool q4) {
    const int64_t r = rows_per_tile(q4);
    return ((N + BN - 1) / BN) * ((M + r - 1) / r);
}

}  // namespace

int tc_tile_m() { return Cfg<true>::ROWS; }

// TMA coordinates and the work-item arithmetic are 32-bit: rows and columns
// below 2^31 - 256.
bool tc_gemm_supported(int64_t M, int64_t N, int64_t K, const void* dx, const void* dw) {
    constexpr int64_t kMax = (1ll << 31) - 256;
    return K % 256 == 0 && M < kMax && N < kMax && K < kMax &&
           ((uintptr_t)dx % 16 == 0) && ((uintptr_t)dw % 16 == 0) && encoder() != nullptr;
}

// dense workspace: a16 [M][K] binary16 | Q8 only: dwT [G][ldt(N)] binary32 and
// w16 [N][K] binary16 (the weight codes widened; Q4 codes are unpacked in
// shared memory instead) | the tail tiles' K-chunk partials (binary32,
// BM x BN each; none without a tail split)
size_t tc_gemm_workspace(int64_t M, int64_t N, int64_t K, bool q4) {
    const int64_t G = K / kGroup;
    size_t w = align16((size_t)M * K * 2);
    if (!q4) w += align16((size_t)G * ldt_of(N) * 4) + align16((size_t)N * K * 2);
    return w + tail_bytes(tail_plan(dense_tile_count(M, N, q4), G));
}

cudaError_t launch_tc_gemm(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                           const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                           void* workspace, cudaStream_t s) {
    const int64_t G = K / kGroup, ldt = ldt_of(N);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    __half* a16 = reinterpret_cast<__half*>(ws);
    size_t off = align16((size_t)M * K * 2);
    widen_rows_kernel<<<widen_grid(M * (K / 16)), 256, 0, s>>>(qx, dx, M, K, a16, nullptr, nullptr,
                                                               nullptr, 1, 0);
    float* dwt = nullptr;
    __half* w16 = nullptr;
    if (!q4) {
        dwt = reinterpret_cast<float*>(ws + off);
        off += align16((size_t)G * ldt * 4);
        w16 = reinterpret_cast<__half*>(ws + off);
        off += align16((size_t)N * K * 2);
        widen_rows_kernel<<<widen_grid(N * (K / 16)), 256, 0, s>>>(
            static_cast<const int8_t*>(qw), nullptr, N, K, w16, nullptr, nullptr, nullptr, 1, 0);
        transpose_scales_kernel<<<dim3((unsigned)(ldt / 64), (unsigned)((G + 31) / 32)), 256, 0, s>>>(
            dw, N, G, dwt, ldt);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb, mdx, mdw;
    const bool maps = q4 ? make_maps<true>(&ma, &mb, &mdx, &mdw, a16, qw, dx, dw, M, N, 0, K)
                         : make_maps<false>(&ma, &mb, &mdx, &mdw, a16, w16, dx, dwt, M, N, ldt, K);
    if (!maps) return cudaErrorInvalidValue;
    const int n_tiles = (int)((N + BN - 1) / BN);
    const int64_t tiles = dense_tile_count(M, N, q4);
    const TailPlan tp = tail_plan(tiles, G);
    const int64_t units = tp.full + tp.tail * tp.split;
    const int64_t ctas = units < sm_count() ? units : sm_count();
    GroupedArgs ga{};
    float* part = reinterpret_cast<float*>(ws + off);
    const TailArgs ta{(int)tp.full, tp.split, part};
    e = q4 ? launch_kernel<true, false>((int)ctas, ma, mb, mdx, mdw, y, M, N, K, ldy, ga, n_tiles, (int)units, ta, s)
           : launch_kernel<false, false>((int)ctas, ma, mb, mdx, mdw, y, M, N, K, ldy, ga, n_tiles, (int)units, ta, s);
    if (e != cudaSuccess || tp.tail == 0) return e;
    const int64_t elems = tp.tail * BM * BN;
    tail_reduce_kernel<<<widen_grid(elems), 256, 0, s>>>(part, (int)tp.full, tp.split, (int)tp.tail,
                                                         n_tiles, rows_per_tile(q4), M, N, y, ldy);
    return cudaGetLastError();
}

// MoE workspace after the routing tables: a16 [P][K] binary16 and dxg [P][G]
// binary32 (gathered activation rows and scales in expert order), and the
// m-tile table (at most P / rows + E tiles, 16 bytes each).
size_t tc_grouped_workspace(int64_t P, int64_t N, int64_t K, int32_t E) {
    (void)N;
    const int64_t G = K / kGroup;
    return align16((size_t)P * K * 2) + align16((size_t)P * G * 4) +
           (size_t)(P / Cfg<true>::ROWS + E + 1) * 16;
}

cudaError_t launch_tc_grouped(const int8_t* qx, const float* dx, int64_t P, int64_t N, int64_t K,
                              const uint8_t* qw4, const uint16_t* dw, float* y, int32_t E,
                              int32_t topk, int32_t x_row_mode, const int32_t* perm,
                              const int32_t* offsets, const int32_t* tile_offsets,
                              void* workspace, cudaStream_t s) {
    const int64_t G = K / kGroup;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    __half* a16 = reinterpret_cast<__half*>(ws);
    float* dxg = reinterpret_cast<float*>(ws + align16((size_t)P * K * 2));
    int4* info = reinterpret_cast<int4*>(ws + align16((size_t)P * K * 2) + align16((size_t)P * G * 4));
    // gather + widen the routed rows (count read on the device: offsets[E])
    widen_rows_kernel<<<widen_grid(P * (K / 16)), 256, 0, s>>>(qx, dx, P, K, a16, dxg, perm,
                                                               offsets + E, topk, x_row_mode);
    tile_info_kernel<<<(E + 255) / 256, 256, 0, s>>>(offsets, tile_offsets, E, Cfg<true>::ROWS, info);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb, mdx, mdw;
    if (!make_maps<true>(&ma, &mb, &mdx, &mdw, a16, qw4, dxg, dw, P, (int64_t)E * N, 0, K))
        return cudaErrorInvalidValue;
    const int n_tiles = (int)((N + BN - 1) / BN);
    GroupedArgs ga{perm, tile_offsets, info, E, N};
    return launch_kernel<true, true>(sm_count(), ma, mb, mdx, mdw, y, P, N, K, N, ga, n_tiles, 0,
                                     TailArgs{0, 1, nullptr}, s);
}

unsigned int read_and_clear_tc_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    cudaMemcpyToSymbol(g_tc_error, &z, sizeof z);
    return v;
}

}  // namespace qg
