// Internal launchers of the CUDA library (not part of the C ABI).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace qg {

// SM count of the current device (cached per device).
int sm_count();

// Raise a kernel's dynamic shared-memory limit once per device.
cudaError_t ensure_smem_attr(const void* func, int bytes, int slot);

struct GatherArgs {
    const int32_t* perm;          // routed pair indices grouped by expert
    const int32_t* offsets;       // [E+1] first position of each expert in perm
    const int32_t* tile_offsets;  // [E+1] first m-tile of each expert
    int32_t E;
    int32_t topk;
    int32_t x_row_mode;
};

cudaError_t launch_quantize_act_q8(const float* x, int64_t M, int64_t K, int64_t ldx,
                                   int8_t* qx, float* dx, cudaStream_t s);
cudaError_t launch_quantize_weight(const float* w, int64_t N, int64_t K, void* qw,
                                   uint16_t* dw, bool q4, cudaStream_t s);

int gemv_split(int64_t M, int64_t N, int64_t K, bool q4, int sm, int R);
// Q8 GEMV from binary32 activations quantized in each block (M <= 8);
// cudaErrorInvalidValue when x's codes and scales exceed a block's shared memory.
cudaError_t launch_gemv_fx(const float* x, int64_t ldx, int64_t M, int64_t N, int64_t K, const void* qw,
                           const uint16_t* dw, float* y, int64_t ldy, cudaStream_t s);
cudaError_t launch_gemv(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                        const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                        cudaStream_t s);

int mma_tile_m();
cudaError_t launch_mma_gemm(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                            const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                            cudaStream_t s);
cudaError_t launch_mma_grouped(const int8_t* qx, const float* dx, int64_t P, int64_t N,
                               int64_t K, const uint8_t* qw4, const uint16_t* dw, float* y,
                               const GatherArgs& ga, cudaStream_t s);

bool tc_gemm_supported(int64_t M, int64_t N, int64_t K, const void* dx, const void* dw);
size_t tc_gemm_workspace(int64_t M, int64_t N, int64_t K, bool q4);
cudaError_t launch_tc_gemm(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                           const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                           void* workspace, cudaStream_t s);
unsigned int read_and_clear_tc_error();
// Test-only: cycles a tensor-core pipeline wait may last (<= 0: the default).
cudaError_t set_wait_limit(long long cycles);
int tc_tile_m();
size_t tc_grouped_workspace(int64_t P, int64_t N, int64_t K, int32_t E);
// Where the m-tile table lies in that workspace (the routing kernel fills it).
int4* tc_grouped_tile_table(void* workspace, int64_t P, int64_t K);
cudaError_t launch_tc_grouped(const int8_t* qx, const float* dx, int64_t P, int64_t N, int64_t K,
                              const uint8_t* qw4, const uint16_t* dw, float* y, int32_t E,
                              int32_t topk, int32_t x_row_mode, const int32_t* perm,
                              const int32_t* offsets, const int32_t* tile_offsets,
                              void* workspace, cudaStream_t s);

// Routing: counts/offsets/perm (+ m-tile offsets for tile height bm when
// tile_offsets != nullptr; + the tensor-core GEMM's m-tile table when
// tile_table != nullptr; + zeroing of unrouted rows of y when y != nullptr).
cudaError_t launch_moe_route(const int32_t* topk_ids, int64_t T, int32_t topk, int32_t E,
                             int32_t* counts, int32_t* offsets, int32_t* perm,
                             int32_t* tile_offsets, int bm, int4* tile_table, float* y, int64_t N,
                             int32_t* d_err, cudaStream_t s);

// MoE steps around the grouped GEMM.
cudaError_t launch_swiglu_quant(const float* gu, int64_t P, int64_t F, int64_t ldgu, int8_t* qh,
                                float* dh, cudaStream_t s);
cudaError_t launch_combine(const float* y, const float* w, int64_t T, int topk, int64_t N,
                           float* out, cudaStream_t s);

// GGUF interleaved Q8_0 / Q4_0 blocks -> planar codes + binary16 scales.
cudaError_t launch_gguf_import(const uint8_t* blocks, int64_t N, int64_t K, void* q, uint16_t* d,
                               bool q4, cudaStream_t s);

// Split-K attention merge.
int splitk_merge_max_splits();
cudaError_t launch_splitk_merge(const float* m, const float* l, const float* acc, int S, int64_t R,
                                int64_t D, float* out, float* lse, cudaStream_t s);

// 3-bit Walsh-Hadamard + Lloyd-Max KV codec.
void kv3_codebook(float* levels, float* thresholds);
cudaError_t launch_kv3_encode(const float* x, int64_t T, int D, int64_t ldx, uint32_t* codes,
                              float* scales, cudaStream_t s);
cudaError_t launch_kv3_decode(const uint32_t* codes, const float* scales, int64_t T, int D,
                              float* x, int64_t ldx, cudaStream_t s);

// Test-only group-dot readout (qgemm_debug_group_dots).
cudaError_t launch_fill_ones(float* v, int64_t n, cudaStream_t s);
cudaError_t launch_one_hot_scales(uint16_t* dw, int64_t N, int64_t G, int64_t g, cudaStream_t s);
cudaError_t launch_scatter_group(const float* y, int64_t M, int64_t N, int64_t G, int64_t g,
                                 int32_t* S, cudaStream_t s);

}  // namespace qg
