// Internal helpers of the CUDA library (not part of the C ABI).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace qg {

constexpr int kGroup = 32;  // elements per quantization group along K

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ldg_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// sum of 4 signed byte products + c
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// sum of 4 (unsigned byte of a) x (signed byte of b) + c
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Four Q4 nibbles (stored value q + 8, one per byte in the low 4 bits of
// each byte) -> four signed bytes q.  t = s ^ 8 is q's low nibble in two's
// complement; bit 3 of t is q's sign, copied into the top 4 bits by the
// multiply (0x08 * 0x1E = 0xF0 per byte, no carry between bytes).
__device__ __forceinline__ uint32_t nib_to_s8(uint32_t s) {
    uint32_t t = s ^ 0x08080808u;
    return t | ((t & 0x08080808u) * 0x1Eu);
}

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

}  // namespace qg
