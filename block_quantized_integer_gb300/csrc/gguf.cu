// Import of GGUF-style interleaved weight blocks into the planar layout the
// kernels read.  The mining-card page ("I wrote a custom CUDA inference
// engine to run Qwen3.5-27B on a $130 mining card", Honest benchmarks) runs
// the same Q8_0 GGUF files as llama.cpp; the GGUF block layout itself is that
// file format's: per 32 weights a binary16 scale followed by the codes,
//   Q8_0: 2 + 32 bytes (int8 codes),
//   Q4_0: 2 + 16 bytes (byte j: element j in the low nibble, element j + 16
//         in the high nibble, each stored as q + 8 -- the planar Q4 layout),
// blocks of a row stored one after the other.  The planar layout keeps codes
// and scales in separate planes so that 16-byte loads and TMA boxes stay
// aligned.  One thread moves one block: reads at 2-byte alignment, writes the
// codes as 16-byte stores.  HBM-bound, run once per weight load.
#include "common.cuh"
#include "kernels.h"

namespace qg {

namespace {

template <bool kQ4>
__global__ void __launch_bounds__(256)
gguf_import_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks, int64_t K,
                   uint8_t* __restrict__ q, uint16_t* __restrict__ d) {
    constexpr int CODE_BYTES = kQ4 ? 16 : 32;
    constexpr int WORDS = (2 + CODE_BYTES) / 2;          // block size in 16-bit words
    const int64_t G = K / kGroup;
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(blocks + b * (2 + CODE_BYTES));
        uint16_t w[WORDS];
#pragma unroll
        for (int i = 0; i < WORDS; ++i) w[i] = src[i];
        const int64_t n = b / G, g = b % G;
        d[b] = w[0];
        uint32_t c[CODE_BYTES / 4];
#pragma unroll
        for (int i = 0; i < CODE_BYTES / 4; ++i)
            c[i] = (uint32_t)w[1 + 2 * i] | ((uint32_t)w[2 + 2 * i] << 16);
        uint8_t* dst = q + n * (kQ4 ? K / 2 : K) + g * CODE_BYTES;
#pragma unroll
        for (int i = 0; i < CODE_BYTES / 16; ++i)
            reinterpret_cast<uint4*>(dst)[i] = make_uint4(c[4 * i], c[4 * i + 1], c[4 * i + 2], c[4 * i + 3]);
    }
}

}  // namespace

cudaError_t launch_gguf_import(const uint8_t* blocks, int64_t N, int64_t K, void* q, uint16_t* d,
                               bool q4, cudaStream_t s) {
    const int64_t n_blocks = N * (K / kGroup);
    int64_t grid = (n_blocks + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    if (q4)
        gguf_import_kernel<true><<<(unsigned)grid, 256, 0, s>>>(blocks, n_blocks, K, (uint8_t*)q, d);
    else
        gguf_import_kernel<false><<<(unsigned)grid, 256, 0, s>>>(blocks, n_blocks, K, (uint8_t*)q, d);
    return cudaGetLastError();
}

}  // namespace qg
