/*
 * qgemm.h -- C ABI of the block-quantized integer GEMM/GEMV library for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation ("I wrote a custom CUDA inference engine to run Qwen3.5-27B on
 * a $130 mining card", Features: a Q8_0 GEMM on int8 dot products for prefill;
 * "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU",
 * Methodology 1: a W4A8 integer decode kernel and a grouped 4-bit GEMM for MoE
 * routing, Methodology 2: group-wise symmetric 4-bit weights with 8-bit
 * activations):
 *
 *   y[m,n] = sum_g dw[n,g] * dx[m,g] * S[m,n,g],
 *   S[m,n,g] = sum_{k = 32g .. 32g+31} qx[m,k] * qw[n,k]     (exact integer)
 *
 * Data layout (all row-major, K contiguous, G = K / 32):
 *   x    float32 [M][ldx]        activations before quantization
 *   qx   int8    [M][K]          quantized activations, q in [-127, 127]
 *   dx   float32 [M][G]          activation scales, d = max|x| / 127
 *   qw   int8    [N][K]          Q8_0 weights, q in [-127, 127]
 *   qw4  uint8   [N][K/2]        Q4_0 weights: in each 16-byte group, byte j
 *                                holds element j (low nibble) and element
 *                                j+16 (high nibble), each stored as q + 8
 *   dw   uint16  [N][G]          weight scales, IEEE binary16 bit patterns
 *   y    float32 [M][ldy]        output
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless stated otherwise; the caller owns
 *     every buffer.  The library allocates nothing, frees nothing and never
 *     synchronizes: work is enqueued on `stream` and runs asynchronously.
 *   - Arguments are validated on the host before anything is enqueued; a
 *     failed check returns a status and enqueues nothing.  Checks: non-null
 *     pointers, K > 0 and K % 32 == 0, N > 0, M >= 0 (M == 0 is a no-op that
 *     returns QG_OK), 16-byte aligned qx/qw/qw4 base pointers, 4-byte aligned
 *     x/dx/y, 2-byte aligned dw, ld >= row length.
 *   - QG_ERR_CUDA is returned when a launch fails (cudaGetLastError after the
 *     launch); errors of the kernels themselves surface on the stream.
 *   - Inputs are assumed finite.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QG_OK = 0,
    QG_ERR_INVALID_ARG = 1,  /* null pointer, bad size, K % 32 != 0, ld too small */
    QG_ERR_ALIGNMENT = 2,    /* a base pointer or leading dimension is misaligned */
    QG_ERR_WORKSPACE = 3,    /* workspace missing or smaller than qgemm_workspace_size() */
    QG_ERR_CUDA = 4,         /* a CUDA call or kernel launch failed */
    QG_ERR_UNSUPPORTED = 5   /* valid request outside what the library handles */
} qg_status;

/* Kernel choice for the *_ex entry points. QG_ALGO_AUTO picks by shape. */
typedef enum {
    QG_ALGO_AUTO = 0,
    QG_ALGO_GEMV = 1,     /* split-K GEMV on dp4a, M <= 8 (decode) */
    QG_ALGO_MMA = 2,      /* warp-level mma.sync int8 tile GEMM, any M */
    QG_ALGO_TCGEN05 = 3   /* tcgen05 tensor-memory GEMM, prefill; K % 256 == 0, needs workspace */
} qg_algo;

/* Workspace sizing: op is one of the QG_OP_* values. */
enum { QG_OP_QGEMM_Q8_0 = 1, QG_OP_QGEMM_Q4_0 = 2, QG_OP_GROUPED_MOE = 3,
       QG_OP_DEBUG_GROUP_DOTS = 4 };

/* Human-readable name of a status. Never NULL. */
const char* qg_status_string(qg_status s);

/* Bytes of device workspace the given call needs (0 if none).  For the dense
 * GEMMs pass M, N, K (T, topk, E ignored): M > 8 with K % 256 == 0 runs on the
 * tensor cores and needs M*K*2 bytes (activation codes widened to binary16)
 * plus (K/32)*ceil32(N)*4 bytes (weight scales transposed to binary32) plus
 * N*K*2 bytes (weight codes widened to binary16), each part padded to 16
 * bytes, plus up to 64 KiB per SM of the current device for
 * the K-chunk partial sums of the output tiles that would leave the last round
 * of the one-CTA-per-SM grid partly empty (0 when the 128 x 128 tile count is a
 * multiple of the SM count); QG_ALGO_TCGEN05 chosen explicitly needs the same
 * for any M (take the size for M = 9 as the floor).  For the MoE GEMM pass K and N and the routing sizes T, topk, E
 * (M ignored).  Workspace pointers must be 16-byte aligned. */
size_t qgemm_workspace_size(int op, int64_t M, int64_t N, int64_t K,
                            int64_t T, int32_t topk, int32_t E);

/* Test-only readout of the exact group dot products
 *   S[m][n][g] = sum_{k = 32g .. 32g+31} qx[m,k] * qw[n,k]
 * as the dense product kernel `algo` forms them (QG_ALGO_AUTO: the kernel the
 * product itself would pick).  The kernel runs once per group g with every
 * activation scale 1 and the weight scales 1 on group g, 0 elsewhere, so its
 * binary32 output is S of that group exactly (|S| <= 32 * 127^2 < 2^19); the
 * result is stored as int32.  No counterpart in the pages: it exists so that a
 * test can compare the integer stage of every kernel bit for bit.
 *   qw: int8 [N][K] (bits 8) or packed uint8 [N][K/2] (bits 4).
 *   S:  int32 [M][N][G], device.
 *   workspace: qgemm_workspace_size(QG_OP_DEBUG_GROUP_DOTS, M, N, K, 0, 0, 0)
 *   bytes, 16-byte aligned (scale planes, one y plane and the product's own
 *   workspace).  Runs 3 G + 1 launches on `stream`; slow by design. */
qg_status qgemm_debug_group_dots(const int8_t* qx, int64_t M, int64_t N, int64_t K,
                                 const void* qw, int bits, int algo, int32_t* S,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Activation quantization, per row m and 32-group g (Methodology 2 of the MoE
 * page: 8-bit activations; Q8 block rule):
 *   d = max_k |x[m,k]| / 127  (one IEEE binary32 division, nearest-even),
 *   q = clamp(round_half_even(x / d), -127, 127)  (binary32 quotient),
 *   d == 0 gives q = 0.
 * x [M][ldx] float32 (ldx >= K), qx [M][K] int8, dx [M][G] float32.
 * Bit-exact: the same bits on every run and every launch shape. */
qg_status quantize_act_q8(const float* x, int64_t M, int64_t K, int64_t ldx,
                          int8_t* qx, float* dx, cudaStream_t stream);

/* Q8_0 weight quantization (Features of the mining-card page: Q8_0 GEMM):
 *   d16 = binary16(max|w| / 127) (nearest-even, saturated to 65504),
 *   q = clamp(round_half_even(w / float(d16)), -127, 127), d16 == 0 gives q = 0.
 * w [N][K] float32 -> qw [N][K] int8, dw [N][G] binary16 bits. */
qg_status quantize_weight_q8_0(const float* w, int64_t N, int64_t K,
                               int8_t* qw, uint16_t* dw, cudaStream_t stream);

/* Q4_0 weight quantization (Methodology 2 of the MoE page: group-wise
 * symmetric 4-bit):  d16 = binary16(max|w| / 7), q = clamp(rhe(w / d16), -8, 7),
 * packed as described for qw4 above.  w [N][K] -> qw4 [N][K/2], dw [N][G]. */
qg_status quantize_weight_q4_0(const float* w, int64_t N, int64_t K,
                               uint8_t* qw4, uint16_t* dw, cudaStream_t stream);

/* Import of weights stored as GGUF-style interleaved blocks (the mining-card
 * page runs the same Q8_0 GGUF files as llama.cpp; the block layout is the
 * GGUF format's): per 32 weights of a row, a binary16 scale followed by the
 * codes -- Q8_0: 2 + 32 bytes of int8; Q4_0: 2 + 16 bytes of nibbles in the
 * qw4 order above -- the K/32 blocks of a row back to back, rows back to back.
 *   blocks: device, [N][K/32][34] (Q8_0) or [N][K/32][18] (Q4_0), 2-byte
 *           aligned;
 *   out:    qw int8 [N][K] / qw4 uint8 [N][K/2] (16-byte aligned), dw
 *           binary16 bits [N][K/32].
 * A pure byte move: the codes and scales come out as stored. */
qg_status import_gguf_q8_0(const uint8_t* blocks, int64_t N, int64_t K, int8_t* qw,
                           uint16_t* dw, cudaStream_t stream);
qg_status import_gguf_q4_0(const uint8_t* blocks, int64_t N, int64_t K, uint8_t* qw4,
                           uint16_t* dw, cudaStream_t stream);

/* Dense Q8_0 x Q8 product (prefill GEMM for large M, decode GEMV for M <= 8):
 * y = sum_g dw * dx * S as above, every S formed exactly before it is scaled,
 * the sum over groups in binary32 (order depends on the kernel; fixed for a
 * given shape and algo, so results are run-to-run deterministic).
 * workspace: at least qgemm_workspace_size() bytes (QG_ERR_WORKSPACE if
 * smaller); NULL/0 when that size is 0. */
qg_status qgemm_q8_0(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                     const int8_t* qw, const uint16_t* dw, float* y, int64_t ldy,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Decode Q8_0 product from binary32 activations, M <= 8 (the activation
 * quantization moved into the GEMV, one launch instead of quantize_act_q8 +
 * qgemm_q8_0): x binary32 [M][ldx] (ldx >= K), every block quantizing all of x
 * into shared memory with quantize_act_q8's rule, then the decode GEMV.  y is
 * bit for bit what quantize_act_q8 followed by qgemm_q8_0 writes.
 * QG_ERR_INVALID_ARG for M outside 1..8 (0 is a no-op), QG_ERR_UNSUPPORTED when
 * M * K * 1.125 bytes exceed 200 KiB (one block's share of x), alignment as
 * qgemm_q8_0 (x: 4 bytes). */
qg_status qgemv_q8_0_f32(const float* x, int64_t M, int64_t K, int64_t ldx, const int8_t* qw,
                         const uint16_t* dw, int64_t N, float* y, int64_t ldy, cudaStream_t stream);

/* Dense Q4_0 x Q8 product: as qgemm_q8_0 with 4-bit weights qw4 [N][K/2]. */
qg_status qgemm_q4_0(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                     const uint8_t* qw4, const uint16_t* dw, float* y, int64_t ldy,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* As qgemm_q8_0 / qgemm_q4_0 with an explicit kernel choice (tests and
 * benchmarks). Returns QG_ERR_UNSUPPORTED when the kernel cannot take the
 * shape (QG_ALGO_GEMV with M > 8). */
qg_status qgemm_q8_0_ex(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                        const int8_t* qw, const uint16_t* dw, float* y, int64_t ldy,
                        void* workspace, size_t workspace_bytes, int algo,
                        cudaStream_t stream);
qg_status qgemm_q4_0_ex(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
                        const uint8_t* qw4, const uint16_t* dw, float* y, int64_t ldy,
                        void* workspace, size_t workspace_bytes, int algo,
                        cudaStream_t stream);

/* MoE routing preparation (Methodology 1 of the MoE page: grouped GEMM for
 * MoE routing).  Pairs p = token * topk + slot, topk_ids [T][topk] int32.
 *   counts [E]    pairs routed to each expert,
 *   offsets [E+1] exclusive prefix sum of counts (offsets[E] = routed pairs),
 *   perm [T*topk] pair indices grouped by expert, (token, slot) order inside
 *                 an expert; entries past offsets[E] are left unspecified.
 * Ids outside [0, E) are not routed: *d_err (device int32) is incremented once
 * per such pair and nothing traps.  Deterministic.  E <= 1024, T*topk < 2^31.
 * T = 0 is valid (topk_ids may then be NULL): counts and offsets are zeroed. */
qg_status moe_route(const int32_t* topk_ids, int64_t T, int32_t topk, int32_t E,
                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* d_err,
                    cudaStream_t stream);

/* Grouped W4A8 MoE GEMM: for every routed pair p with expert e = topk_ids[p],
 *   y[p][:] = x_row(p) * W_e^T,   W_e = Q4_0 weights qw4[e] [N][K/2], dw[e] [N][G],
 * x_row(p) = activation row p / topk (x_row_mode 0, one row per token, rows_x
 * >= T) or row p (x_row_mode 1, one row per pair, rows_x >= T*topk).
 * y [T*topk][N] float32 in (token, slot) order; rows of unrouted pairs (id
 * outside [0, E)) are set to zero and counted in *d_err.  d_err is a device
 * int32 the caller zeroes.  Needs qgemm_workspace_size(QG_OP_GROUPED_MOE, ...)
 * bytes of workspace (16-byte aligned). */
qg_status grouped_qgemm_moe(const int8_t* qx, const float* dx, int64_t rows_x, int64_t K,
                            const int32_t* topk_ids, int64_t T, int32_t topk,
                            int32_t x_row_mode, const uint8_t* qw4, const uint16_t* dw,
                            int32_t E, int64_t N, float* y, int32_t* d_err,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* SwiGLU between the MoE gate/up and down products, re-quantized for the
 * down product (Methodology 1 of the MoE page: 8-bit activations into the
 * W4A8 grouped GEMM; the pages do not spell the activation out, the usual
 * gated one is taken):
 *   h[p, j] = silu(gu[p, j]) * gu[p, F + j],  silu(v) = v / (1 + exp(-v)),
 * evaluated in binary32 (expf, a correctly rounded reciprocal and products),
 * then per row p and 32-group the activation rule of quantize_act_q8, the
 * quotient h / d taken as h times the correctly rounded reciprocal of d.
 *   gu: float32 [P][ldgu], ldgu >= 2F, gate in columns [0, F), up in [F, 2F)
 *       (the fused gate/up output of grouped_qgemm_moe);
 *   qh: int8 [P][F] (16-byte aligned), dh: float32 [P][F/32].  F % 32 == 0.
 * Codes agree with a binary64 evaluation of h except where h / d lies within
 * a few binary32 rounding errors of a half-integer. */
qg_status moe_swiglu_quant(const float* gu, int64_t P, int64_t F, int64_t ldgu,
                           int8_t* qh, float* dh, cudaStream_t stream);

/* Router-weighted combine of the routed rows back into token rows:
 *   out[t][n] = sum_{s = 0 .. topk-1} w[t][s] * y[t * topk + s][n],
 * summed in slot order with binary32 FMAs (deterministic).  y float32
 * [T*topk][N] in (token, slot) order (the down output of grouped_qgemm_moe;
 * unrouted pairs hold zero rows), w float32 [T][topk], out float32 [T][N]. */
qg_status moe_combine(const float* y, const float* w, int64_t T, int32_t topk, int64_t N,
                      float* out, cudaStream_t stream);

/* Split-K attention merge (the mining-card page, Implementation challenges 3:
 * split-K FlashAttention partials merged with the log-sum-exp identity):
 * for each row r (one head, one query) and split s with running max m_s,
 * sum of exponentials l_s and unnormalised output acc_s,
 *   m = max_s m_s,  l = sum_s exp(m_s - m) * l_s,  o = sum_s exp(m_s - m) * acc_s,
 *   out[r] = o / l,  lse[r] = m + log(l),
 * in binary32: the outputs summed over the splits in index order and l in a
 * fixed order, so the result is deterministic.  Empty
 * splits (m_s = -inf, l_s = 0) contribute nothing; a row with only empty
 * splits gives out = 0 and lse = -inf.
 *   m, l: float32 [S][R];  acc: float32 [S][R][D];  out: float32 [R][D];
 *   lse: float32 [R] or NULL.  1 <= S <= 64. */
qg_status attn_splitk_merge(const float* m, const float* l, const float* acc, int32_t S,
                            int64_t R, int64_t D, float* out, float* lse, cudaStream_t stream);

/* 3-bit KV-cache codec (the mining-card page, Features: a 3-bit Walsh-Hadamard +
 * Lloyd-Max KV cache; the pages name the steps only, the reading taken is):
 *   y = H x / sqrt(D), H the Sylvester-ordered Hadamard matrix of order D;
 *   s = sqrt(mean_j y_j^2) (binary32);
 *   code_j = number of thresholds t_k <= y_j / s (0..7; all 0 when s = 0;
 *            the codebook is symmetric about 0 and an exact tie on the
 *            negative side goes to the level of larger magnitude),
 *            t_k = (l_k + l_{k+1}) / 2 over the 8 Lloyd-Max levels l_0 < .. < l_7
 *            of the standard normal distribution (qg_kv3_codebook);
 *   decode: x^ = H (s * l[code]) / sqrt(D).
 * Codes of a vector: 3 bit planes, 3 D / 32 uint32 words; word b * (D/32) + e,
 * bit L holds bit b of the code of element L * (D/32) + e.  D = 64, 128 or 256.
 *   x: float32 [T][ldx] (ldx >= D);  codes: uint32 [T][3 D / 32];  scales: float32 [T].
 * Encode decisions are taken in binary32: z = H x unnormalised, then
 * |z_j| against sqrt(sum z^2) * (t_k / sqrt(D)) for the positive thresholds
 * and the sign of z_j (the same test as y_j / s against t_k for s > 0);
 * s = sqrt(sum z^2) / D.  Codes can therefore differ
 * from an exact evaluation only where y_j / s lies within binary32 rounding of
 * a threshold. */
qg_status kv3_encode(const float* x, int64_t T, int32_t D, int64_t ldx, uint32_t* codes,
                     float* scales, cudaStream_t stream);
qg_status kv3_decode(const uint32_t* codes, const float* scales, int64_t T, int32_t D, float* x,
                     int64_t ldx, cudaStream_t stream);
/* The 8 levels and 7 thresholds in use (HOST arrays), computed once by Lloyd's
 * iteration in binary64 and rounded to binary32. */
void qg_kv3_codebook(float* levels, float* thresholds);

/* grouped_qgemm_moe for callers that cannot allocate device memory: the same
 * arguments minus the workspace.  The product always runs on the warp-level
 * MMA kernel (grouped_qgemm_moe takes the tensor-core kernel when K % 256 == 0),
 * so its y agrees with grouped_qgemm_moe's within the parity tolerance rather
 * than bit for bit.  Errors are grouped_qgemm_moe's, except that E > 1024 or
 * T * topk > 65536 return QG_ERR_UNSUPPORTED (the scratch array's limits).
 * (No counterpart in the pages this library follows: it exists for callers
 * such as a serving process whose device memory is reserved up front by its
 * own pool allocator and that may not call cudaMalloc while running, or a
 * plugin host that passes in buffers but grants no allocation rights.)
 * The routing scratch lives in a fixed array inside the library, held on every
 * GPU that loads it until the process exits: at most 65536 routed pairs
 * (T * topk) and 1024 experts, about 270 KiB; larger requests return
 * QG_ERR_UNSUPPORTED before anything is enqueued.  The call allocates and
 * frees nothing.  Every call rewrites the scratch it reads, so nothing in it
 * needs zeroing (d_err is still zeroed by the caller).  All calls share the one
 * array: calls that overlap on the GPU (unordered streams) race on it.  The
 * first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture. */
qg_status grouped_qgemm_moe_noalloc(const int8_t* qx, const float* dx, int64_t rows_x, int64_t K,
                                    const int32_t* topk_ids, int64_t T, int32_t topk,
                                    int32_t x_row_mode, const uint8_t* qw4, const uint16_t* dw,
                                    int32_t E, int64_t N, float* y, int32_t* d_err,
                                    cudaStream_t stream);

/* Number of streaming multiprocessors of the current device (0 on error). */
int qg_device_sm_count(void);

/* Test-only (no counterpart in the pages): the number of SM clock cycles a
 * pipeline wait of the tensor-core kernels may last on the current device
 * before the kernel gives up (sets bit 0 of the device error word, drains its
 * own copies and MMAs, frees tensor memory and returns without writing its
 * tiles).  cycles <= 0 restores the default, about 2 s.  A blocking copy to
 * the device; it exists so that tests can make a wait run out without
 * withholding any arrival. */
qg_status qg_debug_set_wait_limit(long long cycles);

/* Device error word of the tensor-core kernels on the current device, then
 * cleared: 0 = none, bit 0 = a pipeline wait gave up (the kernel abandoned its
 * tile without writing it, after draining its own copies and freeing tensor
 * memory).  Synchronizes with the device (a blocking copy). */
unsigned int qg_device_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H */
