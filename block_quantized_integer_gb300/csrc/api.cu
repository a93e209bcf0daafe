// C ABI of the library: argument validation on the host, then kernel launches
// on the caller's stream.  See include/qgemm.h for the contract of each entry.
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "../../include/qgemm.h"
#include "kernels.h"

namespace qg {

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = v;
    }
    return cached[dev];
}

cudaError_t ensure_smem_attr(const void* func, int bytes, int slot) {
    static int done[64][16] = {{0}};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || slot < 0 || slot >= 16) return cudaErrorInvalidValue;
    if (done[dev][slot] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[dev][slot] = bytes;
    return e;
}

}  // namespace qg

namespace {

constexpr int64_t kGroup = 32;

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

qg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QG_OK : QG_ERR_CUDA; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// MoE workspace: counts [E], offsets [E+1], tile_offsets [E+1], perm [P], int32.
struct MoeWs {
    size_t counts, offsets, tiles, perm, total;
};
MoeWs moe_ws(int64_t P, int32_t E) {
    MoeWs w{};
    size_t o = 0;
    w.counts = o;  o = align_up(o + 4 * (size_t)E, 16);
    w.offsets = o; o = align_up(o + 4 * (size_t)(E + 1), 16);
    w.tiles = o;   o = align_up(o + 4 * (size_t)(E + 1), 16);
    w.perm = o;    o = align_up(o + 4 * (size_t)P, 16);
    w.total = o;
    return w;
}

qg_status check_dense(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                      const void* qw, const uint16_t* dw, float* y, int64_t ldy) {
    if (M < 0 || N <= 0 || K <= 0 || K % kGroup != 0) return QG_ERR_INVALID_ARG;
    if (M == 0) return QG_OK;
    if (!qx || !dx || !qw || !dw || !y) return QG_ERR_INVALID_ARG;
    if (ldy < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(qx) || !aligned16(qw) || ((uintptr_t)y & 3u)) return QG_ERR_ALIGNMENT;
    if (!aligned16(dx) && ((uintptr_t)dx & 3u)) return QG_ERR_ALIGNMENT;
    if ((uintptr_t)dw & 1u) return QG_ERR_ALIGNMENT;
    return QG_OK;
}

// Dense products with M > 8 run on the tcgen05 kernel when K % 256 == 0 and
// the scale planes are 16-byte aligned (TMA boxes), else on the warp-MMA one.
bool use_tc(int64_t M, int64_t N, int64_t K, const void* dx, const void* dw) {
    return M > 8 && qg::tc_gemm_supported(M, N, K, dx, dw);
}

qg_status dense(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                const void* qw, bool q4, const uint16_t* dw, float* y, int64_t ldy,
                void* ws, size_t ws_bytes, int algo, cudaStream_t s) {
    qg_status st = check_dense(qx, dx, M, N, K, qw, dw, y, ldy);
    if (st != QG_OK || M == 0) return st;
    if (algo == QG_ALGO_AUTO) {
        if (M <= 8) algo = QG_ALGO_GEMV;
        else if (use_tc(M, N, K, dx, dw)) algo = QG_ALGO_TCGEN05;
        else algo = QG_ALGO_MMA;
    }
    switch (algo) {
        case QG_ALGO_GEMV:
            if (M > 8) return QG_ERR_UNSUPPORTED;
            return from_cuda(qg::launch_gemv(qx, dx, M, N, K, qw, q4, dw, y, ldy, s));
        case QG_ALGO_MMA:
            return from_cuda(qg::launch_mma_gemm(qx, dx, M, N, K, qw, q4, dw, y, ldy, s));
        case QG_ALGO_TCGEN05:
            if (!qg::tc_gemm_supported(M, N, K, dx, dw)) return QG_ERR_UNSUPPORTED;
            if (!ws || ws_bytes < qg::tc_gemm_workspace(M, N, K, q4) || !aligned16(ws))
                return QG_ERR_WORKSPACE;
            return from_cuda(qg::launch_tc_gemm(qx, dx, M, N, K, qw, q4, dw, y, ldy, ws, s));
        default:
            return QG_ERR_INVALID_ARG;
    }
}

}  // namespace

extern "C" {

const char* qg_status_string(qg_status s) {
    switch (s) {
        case QG_OK: return "QG_OK";
        case QG_ERR_INVALID_ARG: return "QG_ERR_INVALID_ARG";
        case QG_ERR_ALIGNMENT: return "QG_ERR_ALIGNMENT";
        case QG_ERR_WORKSPACE: return "QG_ERR_WORKSPACE";
        case QG_ERR_CUDA: return "QG_ERR_CUDA";
        case QG_ERR_UNSUPPORTED: return "QG_ERR_UNSUPPORTED";
        default: return "QG_ERR_UNKNOWN";
    }
}

int qg_device_sm_count(void) { return qg::sm_count(); }

unsigned int qg_device_error(void) { return qg::read_and_clear_tc_error(); }

qg_status qg_debug_set_wait_limit(long long cycles) { return from_cuda(qg::set_wait_limit(cycles)); }

// The grouped product runs on the tensor cores when K % 256 == 0 (TMA scale
// boxes) and the expert weight planes (E * N rows) stay within 32-bit TMA
// coordinates, else on the warp-MMA kernel.
bool moe_use_tc(int64_t K, int32_t E, int64_t N) {
    return K > 0 && K % 256 == 0 && (int64_t)E * N < (1ll << 31) - 256;
}

// Debug group-dot workspace: dx = 1 [M][G] f32 | dw one-hot [N][G] binary16 |
// y [M][N] f32 | the dense product's workspace (sized for any algo).
struct DebugWs {
    size_t dx, dw, y, prod, total;
};
DebugWs debug_ws(int64_t M, int64_t N, int64_t K) {
    DebugWs w{};
    const int64_t G = K / kGroup;
    size_t o = 0;
    w.dx = o;   o = align_up(o + 4 * (size_t)(M * G), 16);
    w.dw = o;   o = align_up(o + 2 * (size_t)(N * G), 16);
    w.y = o;    o = align_up(o + 4 * (size_t)(M * N), 16);
    w.prod = o;
    if (K % 256 == 0) {       // either weight format (their tiles, hence tail splits, differ)
        const int64_t m = M > 9 ? M : 9;
        const size_t q8 = qg::tc_gemm_workspace(m, N, K, false), q4 = qg::tc_gemm_workspace(m, N, K, true);
        o += q8 > q4 ? q8 : q4;
    }
    w.total = o;
    return w;
}

size_t qgemm_workspace_size(int op, int64_t M, int64_t N, int64_t K, int64_t T, int32_t topk,
                            int32_t E) {
    if (op == QG_OP_GROUPED_MOE) {
        if (T < 0 || topk <= 0 || E <= 0 || T > ((1ll << 31) - 1) / topk) return 0;
        size_t w = moe_ws(T * topk, E).total;
        if (moe_use_tc(K, E, N) && N > 0) w += qg::tc_grouped_workspace(T * topk, N, K, E);
        return w;
    }
    if (op == QG_OP_DEBUG_GROUP_DOTS) {
        if (M <= 0 || N <= 0 || K <= 0 || K % kGroup != 0) return 0;
        return debug_ws(M, N, K).total;
    }
    if (op == QG_OP_QGEMM_Q8_0 || op == QG_OP_QGEMM_Q4_0) {
        // the tensor-core path widens the activation codes to binary16 first
        if (M > 8 && K > 0 && K % 256 == 0)
            return qg::tc_gemm_workspace(M, N, K, op == QG_OP_QGEMM_Q4_0);
        return 0;
    }
    return 0;
}

qg_status quantize_act_q8(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qx,
                          float* dx, cudaStream_t stream) {
    if (M < 0 || K <= 0 || K % kGroup != 0 || ldx < K) return QG_ERR_INVALID_ARG;
    if (M == 0) return QG_OK;
    if (!x || !qx || !dx) return QG_ERR_INVALID_ARG;
    if (!aligned16(qx) || ((uintptr_t)x & 3u) || ((uintptr_t)dx & 3u)) return QG_ERR_ALIGNMENT;
    return from_cuda(qg::launch_quantize_act_q8(x, M, K, ldx, qx, dx, stream));
}

static qg_status quantize_weight(const float* w, int64_t N, int64_t K, void* q, uint16_t* dw,
                                 bool q4, cudaStream_t stream) {
    if (N < 0 || K <= 0 || K % kGroup != 0) return QG_ERR_INVALID_ARG;
    if (N == 0) return QG_OK;
    if (!w || !q || !dw) return QG_ERR_INVALID_ARG;
    if (!aligned16(q) || ((uintptr_t)w & 3u) || ((uintptr_t)dw & 1u)) return QG_ERR_ALIGNMENT;
    return from_cuda(qg::launch_quantize_weight(w, N, K, q, dw, q4, stream));
}

qg_status quantize_weight_q8_0(const float* w, int64_t N, int64_t K, int8_t* qw, uint16_t* dw,
                               cudaStream_t stream) {
    return quantize_weight(w, N, K, qw, dw, false, stream);
}

qg_status quantize_weight_q4_0(const float* w, int64_t N, int64_t K, uint8_t* qw4, uint16_t* dw,
                               cudaStream_t stream) {
    return quantize_weight(w, N, K, qw4, dw, true, stream);
}

qg_status qgemm_q8_0(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                     const int8_t* qw, const uint16_t* dw, float* y, int64_t ldy,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return dense(qx, dx, M, N, K, qw, false, dw, y, ldy, workspace, workspace_bytes,
                 QG_ALGO_AUTO, stream);
}

qg_status qgemv_q8_0_f32(const float* x, int64_t M, int64_t K, int64_t ldx, const int8_t* qw,
                         const uint16_t* dw, int64_t N, float* y, int64_t ldy, cudaStream_t stream) {
    if (M < 0 || M > 8 || N <= 0 || K <= 0 || K % kGroup != 0) return QG_ERR_INVALID_ARG;
    if (M == 0) return QG_OK;
    if (!x || !qw || !dw || !y || ldx < K || ldy < N) return QG_ERR_INVALID_ARG;
    if (((uintptr_t)x & 3u) || !aligned16(qw) || ((uintptr_t)y & 3u) || ((uintptr_t)dw & 1u))
        return QG_ERR_ALIGNMENT;
    if (M * K + (M * K) / 8 > (int64_t)200 * 1024) return QG_ERR_UNSUPPORTED;
    return from_cuda(qg::launch_gemv_fx(x, ldx, M, N, K, qw, dw, y, ldy, stream));
}

qg_status qgemm_q4_0(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                     const uint8_t* qw4, const uint16_t* dw, float* y, int64_t ldy,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return dense(qx, dx, M, N, K, qw4, true, dw, y, ldy, workspace, workspace_bytes,
                 QG_ALGO_AUTO, stream);
}

qg_status qgemm_q8_0_ex(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                        const int8_t* qw, const uint16_t* dw, float* y, int64_t ldy,
                        void* workspace, size_t workspace_bytes, int algo,
                        cudaStream_t stream) {
    return dense(qx, dx, M, N, K, qw, false, dw, y, ldy, workspace, workspace_bytes, algo,
                 stream);
}

qg_status qgemm_q4_0_ex(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                        const uint8_t* qw4, const uint16_t* dw, float* y, int64_t ldy,
                        void* workspace, size_t workspace_bytes, int algo,
                        cudaStream_t stream) {
    return dense(qx, dx, M, N, K, qw4, true, dw, y, ldy, workspace, workspace_bytes, algo,
                 stream);
}

qg_status moe_route(const int32_t* topk_ids, int64_t T, int32_t topk, int32_t E,
                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* d_err,
                    cudaStream_t stream) {
    if (T < 0 || topk <= 0 || E <= 0 || E > 1024 || T > ((1ll << 31) - 1) / topk)
        return QG_ERR_INVALID_ARG;
    if ((T > 0 && !topk_ids) || !counts || !offsets || !perm || !d_err) return QG_ERR_INVALID_ARG;
    if (((uintptr_t)topk_ids | (uintptr_t)counts | (uintptr_t)offsets | (uintptr_t)perm |
         (uintptr_t)d_err) & 3u)
        return QG_ERR_ALIGNMENT;
    return from_cuda(qg::launch_moe_route(topk_ids, T, topk, E, counts, offsets, perm, nullptr,
                                          1, nullptr, nullptr, 0, d_err, stream));
}

qg_status grouped_qgemm_moe(const int8_t* qx, const float* dx, int64_t rows_x, int64_t K,
                            const int32_t* topk_ids, int64_t T, int32_t topk,
                            int32_t x_row_mode, const uint8_t* qw4, const uint16_t* dw,
                            int32_t E, int64_t N, float* y, int32_t* d_err, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
    if (T < 0 || topk <= 0 || E <= 0 || E > 1024 || N <= 0 || K <= 0 || K % kGroup != 0 ||
        (x_row_mode != 0 && x_row_mode != 1) || T > ((1ll << 31) - 1) / topk)
        return QG_ERR_INVALID_ARG;
    const int64_t P = T * topk;
    if (rows_x < (x_row_mode ? P : T)) return QG_ERR_INVALID_ARG;
    if (T == 0) return QG_OK;
    if (!qx || !dx || !topk_ids || !qw4 || !dw || !y || !d_err) return QG_ERR_INVALID_ARG;
    if (!aligned16(qx) || !aligned16(qw4) || ((uintptr_t)y & 3u) ||
        ((uintptr_t)dx & 3u) || ((uintptr_t)topk_ids & 3u) || ((uintptr_t)d_err & 3u) ||
        ((uintptr_t)dw & 1u))
        return QG_ERR_ALIGNMENT;
    const MoeWs w = moe_ws(P, E);
    const bool tc = moe_use_tc(K, E, N) && ((uintptr_t)dx % 16 == 0) && ((uintptr_t)dw % 16 == 0);
    const size_t need = w.total + (tc ? qg::tc_grouped_workspace(P, N, K, E) : 0);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return QG_ERR_WORKSPACE;
    uint8_t* ws = (uint8_t*)workspace;
    int32_t* counts = (int32_t*)(ws + w.counts);
    int32_t* offsets = (int32_t*)(ws + w.offsets);
    int32_t* tiles = (int32_t*)(ws + w.tiles);
    int32_t* perm = (int32_t*)(ws + w.perm);
    const int bm = tc ? qg::tc_tile_m() : qg::mma_tile_m();
    int4* table = tc ? qg::tc_grouped_tile_table(ws + w.total, P, K) : nullptr;
    cudaError_t e = qg::launch_moe_route(topk_ids, T, topk, E, counts, offsets, perm, tiles, bm,
                                         table, y, N, d_err, stream);
    if (e != cudaSuccess) return QG_ERR_CUDA;
    if (tc)
        return from_cuda(qg::launch_tc_grouped(qx, dx, P, N, K, qw4, dw, y, E, topk, x_row_mode,
                                               perm, offsets, tiles, ws + w.total, stream));
    qg::GatherArgs ga{perm, offsets, tiles, E, topk, x_row_mode};
    return from_cuda(qg::launch_mma_grouped(qx, dx, P, N, K, qw4, dw, y, ga, stream));
}

qg_status qgemm_debug_group_dots(const int8_t* qx, int64_t M, int64_t N, int64_t K,
                                 const void* qw, int bits, int algo, int32_t* S,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (M < 0 || N <= 0 || K <= 0 || K % kGroup != 0 || (bits != 8 && bits != 4))
        return QG_ERR_INVALID_ARG;
    if (M == 0) return QG_OK;
    if (!qx || !qw || !S) return QG_ERR_INVALID_ARG;
    if (!aligned16(qx) || !aligned16(qw) || ((uintptr_t)S & 3u)) return QG_ERR_ALIGNMENT;
    const DebugWs w = debug_ws(M, N, K);
    if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return QG_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* dx = reinterpret_cast<float*>(ws + w.dx);
    uint16_t* dw = reinterpret_cast<uint16_t*>(ws + w.dw);
    float* y = reinterpret_cast<float*>(ws + w.y);
    const int64_t G = K / kGroup;
    if (qg::launch_fill_ones(dx, M * G, stream) != cudaSuccess) return QG_ERR_CUDA;
    for (int64_t g = 0; g < G; ++g) {
        if (qg::launch_one_hot_scales(dw, N, G, g, stream) != cudaSuccess) return QG_ERR_CUDA;
        const qg_status st = dense(qx, dx, M, N, K, qw, bits == 4, dw, y, N, ws + w.prod,
                                   w.total - w.prod, algo, stream);
        if (st != QG_OK) return st;
        if (qg::launch_scatter_group(y, M, N, G, g, S, stream) != cudaSuccess) return QG_ERR_CUDA;
    }
    return QG_OK;
}

qg_status moe_swiglu_quant(const float* gu, int64_t P, int64_t F, int64_t ldgu, int8_t* qh,
                           float* dh, cudaStream_t stream) {
    if (P < 0 || F <= 0 || F % kGroup != 0 || ldgu < 2 * F) return QG_ERR_INVALID_ARG;
    if (P == 0) return QG_OK;
    if (!gu || !qh || !dh) return QG_ERR_INVALID_ARG;
    if (!aligned16(qh) || ((uintptr_t)gu & 3u) || ((uintptr_t)dh & 3u)) return QG_ERR_ALIGNMENT;
    return from_cuda(qg::launch_swiglu_quant(gu, P, F, ldgu, qh, dh, stream));
}

qg_status moe_combine(const float* y, const float* w, int64_t T, int32_t topk, int64_t N,
                      float* out, cudaStream_t stream) {
    if (T < 0 || topk <= 0 || N <= 0) return QG_ERR_INVALID_ARG;
    if (T == 0) return QG_OK;
    if (!y || !w || !out) return QG_ERR_INVALID_ARG;
    if (((uintptr_t)y & 3u) || ((uintptr_t)w & 3u) || ((uintptr_t)out & 3u)) return QG_ERR_ALIGNMENT;
    return from_cuda(qg::launch_combine(y, w, T, topk, N, out, stream));
}

static qg_status import_gguf(const uint8_t* blocks, int64_t N, int64_t K, void* q, uint16_t* dw,
                             bool q4, cudaStream_t stream) {
    if (N < 0 || K <= 0 || K % kGroup != 0) return QG_ERR_INVALID_ARG;
    if (N == 0) return QG_OK;
    if (!blocks || !q || !dw) return QG_ERR_INVALID_ARG;
    if (((uintptr_t)blocks & 1u) || !aligned16(q) || ((uintptr_t)dw & 1u)) return QG_ERR_ALIGNMENT;
    return from_cuda(qg::launch_gguf_import(blocks, N, K, q, dw, q4, stream));
}

qg_status import_gguf_q8_0(const uint8_t* blocks, int64_t N, int64_t K, int8_t* qw, uint16_t* dw,
                           cudaStream_t stream) {
    return import_gguf(blocks, N, K, qw, dw, false, stream);
}

qg_status import_gguf_q4_0(const uint8_t* blocks, int64_t N, int64_t K, uint8_t* qw4,
                           uint16_t* dw, cudaStream_t stream) {
    return import_gguf(blocks, N, K, qw4, dw, true, stream);
}

qg_status attn_splitk_merge(const float* m, const float* l, const float* acc, int32_t S,
                            int64_t R, int64_t D, float* out, float* lse, cudaStream_t stream) {
    if (S <= 0 || S > qg::splitk_merge_max_splits() || R < 0 || D <= 0) return QG_ERR_INVALID_ARG;
    if (R == 0) return QG_OK;
    if (!m || !l || !acc || !out) return QG_ERR_INVALID_ARG;
    if (((uintptr_t)m | (uintptr_t)l | (uintptr_t)acc | (uintptr_t)out | (uintptr_t)lse) & 3u)
        return QG_ERR_ALIGNMENT;
    return from_cuda(qg::launch_splitk_merge(m, l, acc, S, R, D, out, lse, stream));
}

qg_status kv3_encode(const float* x, int64_t T, int32_t D, int64_t ldx, uint32_t* codes,
                     float* scales, cudaStream_t stream) {
    if (T < 0 || (D != 64 && D != 128 && D != 256) || ldx < D) return QG_ERR_INVALID_ARG;
    if (T == 0) return QG_OK;
    if (!x || !codes || !scales) return QG_ERR_INVALID_ARG;
    if (((uintptr_t)x | (uintptr_t)codes | (uintptr_t)scales) & 3u) return QG_ERR_ALIGNMENT;
    return from_cuda(qg::launch_kv3_encode(x, T, D, ldx, codes, scales, stream));
}

qg_status kv3_decode(const uint32_t* codes, const float* scales, int64_t T, int32_t D, float* x,
                     int64_t ldx, cudaStream_t stream) {
    if (T < 0 || (D != 64 && D != 128 && D != 256) || ldx < D) return QG_ERR_INVALID_ARG;
    if (T == 0) return QG_OK;
    if (!x || !codes || !scales) return QG_ERR_INVALID_ARG;
    if (((uintptr_t)x | (uintptr_t)codes | (uintptr_t)scales) & 3u) return QG_ERR_ALIGNMENT;
    return from_cuda(qg::launch_kv3_decode(codes, scales, T, D, x, ldx, stream));
}

void qg_kv3_codebook(float* levels, float* thresholds) {
    if (levels && thresholds) qg::kv3_codebook(levels, thresholds);
}

}  // extern "C"
