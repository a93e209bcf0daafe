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

// Division of 32-bit unsigned numerators by an invariant divisor d >= 1
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, the unsigned case): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, t = mulhi(m, n) gives
// n / d = (t + ((n - t) >> 1)) >> (l - 1) for every n < 2^32.  Replaces the
// 64-bit software division of a flat index into (row, group) coordinates.
struct FastDiv {
    uint32_t d, m, l;
    __host__ explicit FastDiv(uint32_t div = 1) : d(div), m(0), l(0) {
        if (div > 1) {
            uint32_t bits = 0;
            while ((1ull << bits) < div) ++bits;          // ceil(log2 d)
            l = bits;
            m = (uint32_t)((((1ull << 32) * ((1ull << l) - div)) / div) + 1);
        }
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        if (d == 1) return n;
        const uint32_t t = __umulhi(m, n);
        return (t + ((n - t) >> 1)) >> (l - 1);
    }
};

// Programmatic dependent launch.  A kernel launched with launch_pdl() may start
// while the previous kernel on the stream is still finishing; it must call
// pdl_wait() before it reads anything that kernel may have written (the wait
// returns once the previous grid has completed and its writes are visible; it
// is a no-op when the kernel was launched without the attribute).
// pdl_release() lets the next kernel start launching before this one exits.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_release() {
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

}  // namespace qg
