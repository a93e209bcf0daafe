// grouped_qgemm_moe_noalloc: the grouped W4A8 MoE GEMM for callers that
// cannot allocate device memory.
//
// grouped_qgemm_moe needs a few hundred kilobytes of scratch for its routing
// tables (expert counts, offsets, m-tile offsets, the pair permutation) and
// asks the caller for it.  Some callers have no way to provide it: a serving
// process whose device memory is carved up in advance by its own pool
// allocator and that forbids cudaMalloc once it is running, or a plugin host
// that hands plugins input and output buffers but no allocation rights.  This
// entry point keeps that scratch in a fixed array in the library itself, so
// the call allocates nothing.
//
// The array lives in every GPU that loads the library until the process exits
// (kMaxPairs routed pairs and kMaxExperts experts; about 270 KiB).  Each call
// rewrites every entry it reads before reading it, so nothing has to start at
// zero; the caller's d_err is still the caller's to zero.  All calls share the
// one array: calls whose execution overlaps on the GPU (different streams
// without ordering between them) race on it and give wrong results.
//
// The first call on a device looks up the array's device address with
// cudaGetSymbolAddress (with that device current) and caches it; make that
// first call before any stream capture.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "../../include/qgemm.h"
#include "kernels.h"

namespace {

constexpr int64_t kMaxPairs = 65536;
constexpr int32_t kMaxExperts = 1024;

// counts [E] | offsets [E+1] | tile offsets [E+1] | perm [pairs], int32,
// each part padded to 16 bytes (the same layout as the caller-provided
// workspace of grouped_qgemm_moe).
constexpr size_t kCountsOff = 0;
constexpr size_t kOffsetsOff = (4 * kMaxExperts + 15) / 16 * 16;
constexpr size_t kTilesOff = kOffsetsOff + (4 * (kMaxExperts + 1) + 15) / 16 * 16;
constexpr size_t kPermOff = kTilesOff + (4 * (kMaxExperts + 1) + 15) / 16 * 16;
constexpr size_t kScratchBytes = kPermOff + 4 * kMaxPairs;

static __device__ __align__(256) unsigned char g_moe_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (set up once).
void* scratch_on_current_device(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_moe_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" qg_status grouped_qgemm_moe_noalloc(const int8_t* qx, const float* dx, int64_t rows_x,
                                               int64_t K, const int32_t* topk_ids, int64_t T,
                                               int32_t topk, int32_t x_row_mode,
                                               const uint8_t* qw4, const uint16_t* dw,
                                               int32_t E, int64_t N, float* y, int32_t* d_err,
                                               cudaStream_t stream) {
    if (T < 0 || topk <= 0 || E <= 0 || N <= 0 || K <= 0 || K % 32 != 0 ||
        (x_row_mode != 0 && x_row_mode != 1))
        return QG_ERR_INVALID_ARG;
    // T is bounded before the product is formed, so T * topk cannot overflow
    if (E > kMaxExperts || T > kMaxPairs / topk) return QG_ERR_UNSUPPORTED;
    const int64_t P = T * topk;
    if (rows_x < (x_row_mode ? P : T)) return QG_ERR_INVALID_ARG;
    if (T == 0) return QG_OK;
    if (!qx || !dx || !topk_ids || !qw4 || !dw || !y || !d_err) return QG_ERR_INVALID_ARG;
    if (((uintptr_t)qx & 15u) || ((uintptr_t)qw4 & 15u) || ((uintptr_t)y & 3u) ||
        ((uintptr_t)dx & 3u) || ((uintptr_t)topk_ids & 3u) || ((uintptr_t)d_err & 3u) ||
        ((uintptr_t)dw & 1u))
        return QG_ERR_ALIGNMENT;
    cudaError_t e = cudaSuccess;
    unsigned char* ws = static_cast<unsigned char*>(scratch_on_current_device(&e));
    if (ws == nullptr) return QG_ERR_CUDA;
    int32_t* counts = reinterpret_cast<int32_t*>(ws + kCountsOff);
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + kOffsetsOff);
    int32_t* tiles = reinterpret_cast<int32_t*>(ws + kTilesOff);
    int32_t* perm = reinterpret_cast<int32_t*>(ws + kPermOff);
    e = qg::launch_moe_route(topk_ids, T, topk, E, counts, offsets, perm, tiles,
                             qg::mma_tile_m(), nullptr, y, N, d_err, stream);
    if (e != cudaSuccess) return QG_ERR_CUDA;
    qg::GatherArgs ga{perm, offsets, tiles, E, topk, x_row_mode};
    e = qg::launch_mma_grouped(qx, dx, P, N, K, qw4, dw, y, ga, stream);
    return e == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}
