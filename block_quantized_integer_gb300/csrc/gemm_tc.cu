// Prefill GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// y[m,n] = sum_g dw[n,g] dx[m,g] S[m,n,g] with S the exact integer dot
// product of one 32-group ("I wrote a custom CUDA inference engine to run
// Qwen3.5-27B on a $130 mining card", Features: the Q8_0 GEMM tile path of the
// prefill; "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU",
// Methodology 4: one pass over the whole prompt keeps the GEMM M large).
//
// sm_103a has no integer tcgen05 MMA form, so the int8 codes are widened to
// binary16, where every value in [-127, 127] is exact, and multiplied with
// kind::f16 into binary32 tensor memory: each product is an integer below
// 2^14 and each group sum an integer below 2^19, exact as long as the tensor
// core accumulates a 32-term integer sum without loss (the group-dot tests
// check this bit for bit on extreme groups).
//
// Per CTA: a 128 x 256 output tile, K walked one 32-group at a time.
//   warp 8      TMA producer: int8 A/B tiles, 4 groups per stage, 128-byte
//               swizzle; dx / dw scale tiles every 8 groups.
//   warps 10-11 converters: int8 -> binary16 into the canonical K-major
//               no-swizzle operand layout (8x16-byte core matrices), one
//               32-group per operand buffer, 3 buffers.
//   warp 9      one thread issues two K=16 MMAs per group into one of two
//               256-column TMEM accumulators (first with D overwritten).
//   warps 0-7   epilogue: tcgen05.ld of the group's exact partial, then
//               y += S * (dx * dw) into binary32 registers (thread = row,
//               warpgroup = 128 columns); y is written once at the end.
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

constexpr int BM = 128, BN = 256;
constexpr int GS = 4;                   // groups per int8 TMA stage (128 bytes of K)
constexpr int NS = 2;                   // int8 stages
constexpr int NF = 3;                   // binary16 operand buffers (one group each)
constexpr int SCG = 8;                  // groups per scale stage
constexpr int THREADS = 384;
constexpr int EPI_THREADS = 256;
constexpr int CONV_WARP0 = 10, CONV_WARPS = 2, CONV_THREADS = CONV_WARPS * 32;

constexpr int I8_A_BYTES = BM * GS * 32;             // 16384
constexpr int I8_B_BYTES = BN * GS * 32;             // 32768
constexpr int I8_STAGE = I8_A_BYTES + I8_B_BYTES;    // 49152
constexpr int F16_A_BYTES = BM * 32 * 2;             // 8192
constexpr int F16_B_BYTES = BN * 32 * 2;             // 16384
constexpr int F16_STAGE = F16_A_BYTES + F16_B_BYTES; // 24576
constexpr int SC_DX = BM * SCG * 4;                  // 4096: dx [128][8] f32
constexpr int SC_DW = BN * SCG * 2;                  // 4096: dw [256][8] f16
constexpr int SC_DWF = SCG * BN * 4;                 // 8192: dw [8][256] f32
constexpr int SC_STAGE = SC_DX + SC_DW + SC_DWF;     // 16384

constexpr int OFF_I8 = 0;
constexpr int OFF_F16 = OFF_I8 + NS * I8_STAGE;
constexpr int OFF_SC = OFF_F16 + NF * F16_STAGE;
constexpr int OFF_BAR = OFF_SC + 2 * SC_STAGE;
constexpr int NUM_BARS = 2 * NS + 2 * NF + 3 * 2 + 2 * 2 + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;     // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t TMEM_COLS = 512;     // two 256-column accumulators
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
constexpr uint32_t kSpinLimit = 1u << 22;

struct Bars {
    uint32_t full_i8, empty_i8, full_f16, empty_f16, full_sc, ready_sc, empty_sc, tfull,
        tempty, drain;
};

__device__ __forceinline__ Bars bars_at(uint32_t base) {
    Bars b;
    b.full_i8 = base;
    b.empty_i8 = b.full_i8 + NS * 8;
    b.full_f16 = b.empty_i8 + NS * 8;
    b.empty_f16 = b.full_f16 + NF * 8;
    b.full_sc = b.empty_f16 + NF * 8;
    b.ready_sc = b.full_sc + 16;
    b.empty_sc = b.ready_sc + 16;
    b.tfull = b.empty_sc + 16;
    b.tempty = b.tfull + 16;
    b.drain = b.tempty + 16;
    return b;
}

// Bounded wait.  kWarp: all 32 lanes call it and leave together.
template <bool kWarp>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort) {
    for (uint32_t it = 1;; ++it) {
        bool ok = mbar_try_wait(bar, parity);
        if (kWarp) ok = __all_sync(0xffffffffu, ok);
        if (ok) return true;
        if ((it & 63) == 0) {
            bool ab = *abort != 0;
            if (kWarp) ab = __any_sync(0xffffffffu, ab);
            if (ab) return false;
            if (it > kSpinLimit) {
                *abort = 1;
                atomicOr(&g_tc_error, 1u);
                return false;
            }
        }
    }
}

// 16 int8 -> 16 binary16, exactly: (b ^ 0x80) is b + 128 in [1, 255]; placed
// under the exponent byte 0x64 it reads as 1024 + b + 128; minus 1152 gives b.
__device__ __forceinline__ uint32_t s8x2_to_h2(uint32_t t, uint32_t sel) {
    uint32_t h = __byte_perm(t, 0x64646464u, sel);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}
__device__ __forceinline__ void convert16(const uint4 v, uint4& lo, uint4& hi) {
    const uint32_t a = v.x ^ 0x80808080u, b = v.y ^ 0x80808080u;
    const uint32_t c = v.z ^ 0x80808080u, d = v.w ^ 0x80808080u;
    lo = make_uint4(s8x2_to_h2(a, 0x4140), s8x2_to_h2(a, 0x4342),
                    s8x2_to_h2(b, 0x4140), s8x2_to_h2(b, 0x4342));
    hi = make_uint4(s8x2_to_h2(c, 0x4140), s8x2_to_h2(c, 0x4342),
                    s8x2_to_h2(d, 0x4140), s8x2_to_h2(d, 0x4342));
}

__global__ void __launch_bounds__(THREADS, 1)
tc_gemm_q8_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                  const __grid_constant__ CUtensorMap map_dx, const __grid_constant__ CUtensorMap map_dw,
                  float* __restrict__ y, int64_t M, int64_t N, int64_t K, int64_t ldy, bool vec4) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Bars B = bars_at(sbase + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    const int G = (int)(K / kGroup);
    const int nstages = G / GS;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(B.full_i8 + 8 * i, 1);
            mbar_init(B.empty_i8 + 8 * i, CONV_WARPS);
        }
        for (int i = 0; i < NF; ++i) {
            mbar_init(B.full_f16 + 8 * i, CONV_WARPS);
            mbar_init(B.empty_f16 + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(B.full_sc + 8 * i, 1);
            mbar_init(B.ready_sc + 8 * i, CONV_WARPS);
            mbar_init(B.empty_sc + 8 * i, EPI_THREADS / 32);
            mbar_init(B.tfull + 8 * i, 1);
            mbar_init(B.tempty + 8 * i, EPI_THREADS / 32);
        }
        mbar_init(B.drain, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
        tma_prefetch_desc(&map_dx);
        tma_prefetch_desc(&map_dw);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued_i8 = 0, issued_sc = 0;
            bool ok = true;
            for (int s = 0; s < nstages && ok; ++s) {
                if (s % 2 == 0) {
                    const int sc = s / 2;
                    ok = wait_bar<false>(B.empty_sc + 8 * (sc % 2), ((sc / 2) & 1) ^ 1, abort);
                    if (!ok) break;
                    const uint32_t slot = sbase + OFF_SC + (sc % 2) * SC_STAGE;
                    mbar_expect_tx(B.full_sc + 8 * (sc % 2), SC_DX + SC_DW);
                    tma_load_2d(slot, &map_dx, sc * SCG, m0, B.full_sc + 8 * (sc % 2));
                    tma_load_2d(slot + SC_DX, &map_dw, sc * SCG, n0, B.full_sc + 8 * (sc % 2));
                    issued_sc = sc + 1;
                }
                ok = wait_bar<false>(B.empty_i8 + 8 * (s % NS), ((s / NS) & 1) ^ 1, abort);
                if (!ok) break;
                const uint32_t slot = sbase + OFF_I8 + (s % NS) * I8_STAGE;
                mbar_expect_tx(B.full_i8 + 8 * (s % NS), I8_STAGE);
                tma_load_2d(slot, &map_a, s * GS * 32, m0, B.full_i8 + 8 * (s % NS));
                tma_load_2d(slot + I8_A_BYTES, &map_b, s * GS * 32, n0, B.full_i8 + 8 * (s % NS));
                issued_i8 = s + 1;
            }
            if (!ok) {
                // drain: wait (bounded) for the copies this thread issued
                for (int s = issued_i8 - NS; s < issued_i8; ++s)
                    if (s >= 0) {
                        for (uint32_t it = 0; it < kSpinLimit; ++it)
                            if (mbar_try_wait(B.full_i8 + 8 * (s % NS), (s / NS) & 1)) break;
                    }
                for (int sc = issued_sc - 2; sc < issued_sc; ++sc)
                    if (sc >= 0) {
                        for (uint32_t it = 0; it < kSpinLimit; ++it)
                            if (mbar_try_wait(B.full_sc + 8 * (sc % 2), (sc / 2) & 1)) break;
                    }
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool issued_any = false;
            for (int g = 0; g < G; ++g) {
                const int f = g % NF, b = g % 2;
                if (!wait_bar<false>(B.full_f16 + 8 * f, (g / NF) & 1, abort)) break;
                if (!wait_bar<false>(B.tempty + 8 * b, ((g / 2) & 1) ^ 1, abort)) break;
                tc_fence_after();
                const uint32_t a_s = sbase + OFF_F16 + f * F16_STAGE;
                const uint32_t b_s = a_s + F16_A_BYTES;
                const uint32_t d = tmem_base + (uint32_t)(b * BN);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint64_t ad = smem_desc_noswizzle(a_s + j * 256, 128, 512);
                    const uint64_t bd = smem_desc_noswizzle(b_s + j * 256, 128, 512);
                    mma_f16(d, ad, bd, IDESC, j);
                }
                mma_commit(B.empty_f16 + 8 * f);
                mma_commit(B.tfull + 8 * b);
                issued_any = true;
            }
            if (*abort && issued_any) {
                mma_commit(B.drain);
                for (uint32_t it = 0; it < kSpinLimit; ++it)
                    if (mbar_try_wait(B.drain, 0)) break;
            }
        }
    } else if (warp >= CONV_WARP0) {
        // ------------------------------------------------------------ converters
        const int ct = tid - CONV_WARP0 * 32;
        for (int g = 0; g < G; ++g) {
            const int gi = g % GS, s = g / GS;
            if (gi == 0 && !wait_bar<true>(B.full_i8 + 8 * (s % NS), (s / NS) & 1, abort)) break;
            if (g % SCG == 0) {
                const int sc = g / SCG;
                if (!wait_bar<true>(B.full_sc + 8 * (sc % 2), (sc / 2) & 1, abort)) break;
                uint8_t* slot = smem + OFF_SC + (sc % 2) * SC_STAGE;
                const uint16_t* dw_raw = reinterpret_cast<const uint16_t*>(slot + SC_DX);
                float* dwf = reinterpret_cast<float*>(slot + SC_DX + SC_DW);
                for (int idx = ct; idx < SCG * BN; idx += CONV_THREADS) {
                    const int gg = idx >> 8, col = idx & (BN - 1);
                    dwf[gg * BN + col] = half_bits_to_float(dw_raw[col * SCG + gg]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(B.ready_sc + 8 * (sc % 2));
            }
            const int f = g % NF;
            if (!wait_bar<true>(B.empty_f16 + 8 * f, ((g / NF) & 1) ^ 1, abort)) break;
            const uint8_t* i8 = smem + OFF_I8 + (s % NS) * I8_STAGE;
            uint8_t* f16 = smem + OFF_F16 + f * F16_STAGE;
#pragma unroll 4
            for (int j = 0; j < (BM + BN) * 2 / CONV_THREADS; ++j) {
                const int i = ct + j * CONV_THREADS;
                int row, half;
                const uint8_t* src_tile;
                uint8_t* dst_tile;
                if (i < BM * 2) {
                    row = i & (BM - 1); half = i >> 7;
                    src_tile = i8; dst_tile = f16;
                } else {
                    const int jj = i - BM * 2;
                    row = jj & (BN - 1); half = jj >> 8;
                    src_tile = i8 + I8_A_BYTES; dst_tile = f16 + F16_A_BYTES;
                }
                // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7)
                const int chunk = gi * 2 + half;
                const uint4 v = *reinterpret_cast<const uint4*>(
                    src_tile + row * 128 + ((chunk ^ (row & 7)) << 4));
                uint4 lo, hi;
                convert16(v, lo, hi);
                uint8_t* dst = dst_tile + (row >> 3) * 512 + (half * 2) * 128 + (row & 7) * 16;
                *reinterpret_cast<uint4*>(dst) = lo;
                *reinterpret_cast<uint4*>(dst + 128) = hi;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(B.full_f16 + 8 * f);
                if (gi == GS - 1) mbar_arrive(B.empty_i8 + 8 * (s % NS));
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int wg = tid >> 7, q = warp & 3;
        const int row = q * 32 + lane;
        const int cb = wg * 128;
        float acc[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) acc[i] = 0.f;
        bool ok = true;
        for (int g = 0; g < G && ok; ++g) {
            const int sc = g / SCG, b = g % 2;
            if (g % SCG == 0) ok = wait_bar<true>(B.ready_sc + 8 * (sc % 2), (sc / 2) & 1, abort);
            if (!ok) break;
            ok = wait_bar<true>(B.tfull + 8 * b, (g / 2) & 1, abort);
            if (!ok) break;
            tc_fence_after();
            const uint8_t* slot = smem + OFF_SC + (sc % 2) * SC_STAGE;
            const float dxv = reinterpret_cast<const float*>(slot)[row * SCG + (g % SCG)];
            const float* dwf = reinterpret_cast<const float*>(slot + SC_DX + SC_DW) +
                               (g % SCG) * BN + cb;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + cb);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t s[16];
                tmem_ld16(taddr + c * 16, s);
                tmem_wait_ld();
                if (c == 7) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B.tempty + 8 * b);
                }
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    const float4 w = *reinterpret_cast<const float4*>(dwf + c * 16 + i4 * 4);
                    const int o = c * 16 + i4 * 4;
                    acc[o + 0] = fmaf(__uint_as_float(s[i4 * 4 + 0]), dxv * w.x, acc[o + 0]);
                    acc[o + 1] = fmaf(__uint_as_float(s[i4 * 4 + 1]), dxv * w.y, acc[o + 1]);
                    acc[o + 2] = fmaf(__uint_as_float(s[i4 * 4 + 2]), dxv * w.z, acc[o + 2]);
                    acc[o + 3] = fmaf(__uint_as_float(s[i4 * 4 + 3]), dxv * w.w, acc[o + 3]);
                }
            }
            if (g % SCG == SCG - 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(B.empty_sc + 8 * (sc % 2));
            }
        }
        if (ok && m0 + row < M) {
            float* yr = y + (int64_t)(m0 + row) * ldy + n0 + cb;
            const int64_t ncols = N - (n0 + cb);
            if (vec4 && ncols >= 128) {
#pragma unroll
                for (int i = 0; i < 128; i += 4)
                    *reinterpret_cast<float4*>(yr + i) =
                        make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i < ncols) yr[i] = acc[i];
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

}  // namespace

bool tc_gemm_supported(int64_t M, int64_t N, int64_t K, const void* dx, const void* dw) {
    (void)M; (void)N;
    return K % 256 == 0 && ((uintptr_t)dx % 16 == 0) && ((uintptr_t)dw % 16 == 0) &&
           encoder() != nullptr;
}

cudaError_t launch_tc_gemm(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                           const int8_t* qw, const uint16_t* dw, float* y, int64_t ldy,
                           cudaStream_t s) {
    const int64_t G = K / kGroup;
    CUtensorMap ma, mb, mdx, mdw;
    if (!make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, qx, K, M, K, 128, BM,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, K, N, K, 128, BN,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mdx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dx, G, M, G * 4, SCG, BM,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mdw, CU_TENSOR_MAP_DATA_TYPE_UINT16, dw, G, N, G * 2, SCG, BN,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem_attr((const void*)tc_gemm_q8_kernel, SMEM_BYTES, 9);
    if (e != cudaSuccess) return e;
    const bool vec4 = ((uintptr_t)y % 16 == 0) && (ldy % 4 == 0);
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    tc_gemm_q8_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(ma, mb, mdx, mdw, y, M, N, K, ldy, vec4);
    return cudaGetLastError();
}

unsigned int read_and_clear_tc_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    cudaMemcpyToSymbol(g_tc_error, &z, sizeof z);
    return v;
}

}  // namespace qg
