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
// aligned.  HBM-bound, run once per weight load.
//
// When the block array starts on a 16-byte boundary (32 blocks = 1088 / 576
// bytes, a multiple of 16), a warp moves 32 blocks at a time: 16-byte loads
// into shared memory, then each lane takes one block out of it with 4-byte
// reads and funnel shifts and writes its codes as 16-byte stores (the 32 lanes
// of a warp write 1 KiB / 512 bytes of consecutive codes).  Otherwise, and for
// the last blocks, one thread moves one block with 2-byte reads.
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

template <bool kQ4>
__global__ void __launch_bounds__(256)
gguf_import_vec_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks, int64_t K,
                       uint8_t* __restrict__ q, uint16_t* __restrict__ d) {
    constexpr int CB = kQ4 ? 16 : 32, BB = 2 + CB;        // code bytes, block bytes
    constexpr int CHUNK = 32 * BB, WORDS = CHUNK / 16;    // 32 blocks: 1088 / 576 bytes
    static_assert(CHUNK % 16 == 0, "a chunk of 32 blocks is a whole number of 16-byte words");
    __shared__ __align__(16) uint8_t buf[8][CHUNK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = K / kGroup;
    const int64_t chunks = n_blocks / 32;
    uint8_t* sb = buf[warp];
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(sb);
    // lane's block inside the chunk: the scale at byte off, codes from off + 2
    const int off = lane * BB;
    const int cw0 = (off + 2) >> 2, sh = ((off + 2) & 3) * 8;   // sh is 0 or 16
    for (int64_t c = (int64_t)blockIdx.x * 8 + warp; c < chunks; c += (int64_t)gridDim.x * 8) {
        const uint8_t* src = blocks + c * CHUNK;
#pragma unroll
        for (int i = lane; i < WORDS; i += 32)
            reinterpret_cast<uint4*>(sb)[i] = ldg_nc_v4(src + 16 * i);
        __syncwarp();
        const int64_t b = c * 32 + lane;
        const uint32_t s0 = sw[off >> 2];
        const uint16_t scale = (uint16_t)((off & 3) ? (s0 >> 16) : (s0 & 0xffffu));
        uint32_t cw[CB / 4];
#pragma unroll
        for (int j = 0; j < CB / 4; ++j)
            cw[j] = sh ? __funnelshift_r(sw[cw0 + j], sw[cw0 + j + 1], 16) : sw[cw0 + j];
        __syncwarp();                                       // buffer free for the next chunk
        const int64_t n = b / G, g = b % G;
        d[b] = scale;
        uint4* dst = reinterpret_cast<uint4*>(q + n * (kQ4 ? K / 2 : K) + g * CB);
#pragma unroll
        for (int i = 0; i < CB / 16; ++i) dst[i] = make_uint4(cw[4 * i], cw[4 * i + 1], cw[4 * i + 2], cw[4 * i + 3]);
    }
    // blocks past the last whole chunk: one thread a block, 2-byte reads
    const int64_t tail0 = chunks * 32;
    for (int64_t b = tail0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(blocks + b * BB);
        uint32_t cw[CB / 4];
#pragma unroll
        for (int j = 0; j < CB / 4; ++j) cw[j] = (uint32_t)src[1 + 2 * j] | ((uint32_t)src[2 + 2 * j] << 16);
        const int64_t n = b / G, g = b % G;
        d[b] = src[0];
        uint4* dst = reinterpret_cast<uint4*>(q + n * (kQ4 ? K / 2 : K) + g * CB);
#pragma unroll
        for (int i = 0; i < CB / 16; ++i) dst[i] = make_uint4(cw[4 * i], cw[4 * i + 1], cw[4 * i + 2], cw[4 * i + 3]);
    }
}

}  // namespace

cudaError_t launch_gguf_import(const uint8_t* blocks, int64_t N, int64_t K, void* q, uint16_t* d,
                               bool q4, cudaStream_t s) {
    const int64_t n_blocks = N * (K / kGroup);
    if (((uintptr_t)blocks & 15u) == 0) {
        int64_t grid = (n_blocks / 32 + 7) / 8;
        const int64_t cap = (int64_t)sm_count() * 8;
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
        if (q4)
            gguf_import_vec_kernel<true><<<(unsigned)grid, 256, 0, s>>>(blocks, n_blocks, K, (uint8_t*)q, d);
        else
            gguf_import_vec_kernel<false><<<(unsigned)grid, 256, 0, s>>>(blocks, n_blocks, K, (uint8_t*)q, d);
        return cudaGetLastError();
    }
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
