/*
 * qoracle.c -- plain, slow CPU oracle for block-quantized integer GEMM/GEMV.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark may load this library.  The CUDA
 * library shares no source, header, table or helper with it.
 *
 * What it computes (the method of the pages "I wrote a custom CUDA inference
 * engine to run Qwen3.5-27B on a $130 mining card" -- Features: Q8_0 GEMM on
 * int8 dot products -- and "A 35B Hybrid-Attention Mixture-of-Experts Model on
 * a 6GB 2011 GPU" -- Methodology 1: W4A8 integer multiply-adds and a grouped
 * 4-bit GEMM for MoE routing; Methodology 2: group-wise symmetric 4-bit
 * weights with 8-bit activations):
 *
 *   * weights in groups of 32 along K with one binary16 scale per group,
 *     Q8_0: d = max|w| / 127, q in [-127, 127];
 *     Q4_0: d = max|w| / 7,   q in [-8, 7], two q per byte;
 *   * activations in groups of 32 along K with one binary32 scale per group,
 *     d = max|x| / 127, q in [-127, 127];
 *   * y[m,n] = sum_g dw[n,g] * dx[m,g] * S[m,n,g],
 *     S[m,n,g] = sum_{k in group g} qx[m,k] * qw[n,k]  (an exact integer).
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - scale division is one IEEE binary32 division, q = round-half-even of the
 *     binary32 quotient x / d, then clamped; d == 0 gives q = 0;
 *   - a weight scale is rounded to binary16 (nearest-even, saturated at 65504)
 *     first, and q is computed against the stored binary16 value;
 *   - Q4 packing: byte j (0..15) of a group holds element j in its low nibble
 *     and element j+16 in its high nibble, each stored as q + 8;
 *   - y is summed in binary64 in group order and rounded once to binary32.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off (never -ffast-math), optional
 * -fopenmp: the only parallel loops are over independent output rows.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_GROUP 32

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- binary16 <-> binary32 ------------------------------------------------
 * IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Every finite binary16 value is n * 2^(E-10) for an integer n in [0, 2048)
 * and E = max(exponent, -14); encode finds E from the magnitude, rounds
 * v / 2^(E-10) to the nearest integer (ties to even; the division by a power
 * of two is exact), and lays out the bits. A carry of n to 2048 moves into the
 * exponent field by itself, and past the largest finite value it gives Inf. */
uint16_t orc_f32_to_f16(float f) {
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    double v = fabs((double)f);
    if (isinf(f) || v >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (v == 0.0) return sign;
    int e2;
    frexp(v, &e2);           /* v = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;          /* v in [2^E, 2^(E+1)) */
    if (E < -14) E = -14;
    double n = nearbyint(ldexp(v, 10 - E));   /* round-half-even */
    long field = ((long)(E + 15) << 10) + (long)n - 1024;
    return (uint16_t)(sign | (uint16_t)field);
}

float orc_f16_to_f32(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, fr = h & 0x3ff;
    double v;
    if (e == 0x1f) v = fr ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)fr, -24);
    else v = ldexp((double)(1024 + fr), e - 25);
    return (float)(s ? -v : v);
}

/* ---- quantizers ------------------------------------------------------------ */

static int clamp_int(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* q = clamp(round-half-even(x / d), lo, hi) in binary32; d == 0 gives 0. */
static int quantize_one(float x, float d, int lo, int hi) {
    if (d == 0.0f) return 0;
    float v = x / d;
    return clamp_int((int)rintf(v), lo, hi);
}

static float group_amax(const float* x) {
    float a = 0.0f;
    for (int i = 0; i < ORC_GROUP; ++i) {
        float v = fabsf(x[i]);
        if (v > a) a = v;
    }
    return a;
}

/* Activations: per row m, per 32-group g: d = amax / 127 (binary32), q int8. */
void orc_quantize_act_q8(const float* x, int64_t M, int64_t K, int64_t ldx,
                         int8_t* qx, float* dx) {
    int64_t G = K / ORC_GROUP;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < G; ++g) {
            const float* xg = x + m * ldx + g * ORC_GROUP;
            float d = group_amax(xg) / 127.0f;
            dx[m * G + g] = d;
            for (int i = 0; i < ORC_GROUP; ++i)
                qx[m * K + g * ORC_GROUP + i] = (int8_t)quantize_one(xg[i], d, -127, 127);
        }
    }
}

/* binary16 scale from amax / qmax, saturated to the largest finite value. */
static uint16_t weight_scale(float amax, float qmax) {
    uint16_t h = orc_f32_to_f16(amax / qmax);
    if ((h & 0x7fffu) == 0x7c00u) h = (uint16_t)((h & 0x8000u) | 0x7bffu);
    return h;
}

/* Q8_0 weights: w [N][K] -> qw int8 [N][K], dw binary16 [N][G]. */
void orc_quantize_w_q8_0(const float* w, int64_t N, int64_t K, int8_t* qw, uint16_t* dw) {
    int64_t G = K / ORC_GROUP;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const float* wg = w + n * K + g * ORC_GROUP;
            uint16_t h = weight_scale(group_amax(wg), 127.0f);
            float d = orc_f16_to_f32(h);
            dw[n * G + g] = h;
            for (int i = 0; i < ORC_GROUP; ++i)
                qw[n * K + g * ORC_GROUP + i] = (int8_t)quantize_one(wg[i], d, -127, 127);
        }
    }
}

/* Q4_0 weights: w [N][K] -> qw4 uint8 [N][K/2] (nibble layout above), dw [N][G]. */
void orc_quantize_w_q4_0(const float* w, int64_t N, int64_t K, uint8_t* qw4, uint16_t* dw) {
    int64_t G = K / ORC_GROUP;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const float* wg = w + n * K + g * ORC_GROUP;
            uint16_t h = weight_scale(group_amax(wg), 7.0f);
            float d = orc_f16_to_f32(h);
            dw[n * G + g] = h;
            int q[ORC_GROUP];
            for (int i = 0; i < ORC_GROUP; ++i) q[i] = quantize_one(wg[i], d, -8, 7);
            uint8_t* out = qw4 + n * (K / 2) + g * (ORC_GROUP / 2);
            for (int j = 0; j < ORC_GROUP / 2; ++j)
                out[j] = (uint8_t)((q[j] + 8) | ((q[j + 16] + 8) << 4));
        }
    }
}

/* Element k of a Q4 row (k counts from the start of the row). */
static int q4_at(const uint8_t* row, int64_t k) {
    int64_t g = k / ORC_GROUP, i = k % ORC_GROUP;
    uint8_t b = row[g * (ORC_GROUP / 2) + (i % 16)];
    int nib = (i < 16) ? (b & 0x0f) : (b >> 4);
    return nib - 8;
}

/* ---- group dot products ---------------------------------------------------- */

/* S[m][n][g] = sum_{k in g} qx[m,k] * qw[n,k]; wbits = 8 (int8 rows of K) or 4. */
void orc_group_dots(const int8_t* qx, int64_t M, int64_t N, int64_t K,
                    const void* qw, int wbits, int32_t* S) {
    int64_t G = K / ORC_GROUP;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t g = 0; g < G; ++g) {
                int32_t s = 0;
                for (int i = 0; i < ORC_GROUP; ++i) {
                    int64_t k = g * ORC_GROUP + i;
                    int wv = (wbits == 8) ? ((const int8_t*)qw)[n * K + k]
                                          : q4_at((const uint8_t*)qw + n * (K / 2), k);
                    s += (int32_t)qx[m * K + k] * wv;
                }
                S[(m * N + n) * G + g] = s;
            }
}

/* ---- y = sum_g dw * dx * S --------------------------------------------------- */

/* Columns [n0, n1) of one output row: y[n] from activation row (qxr, dxr) and
 * the weight rows of one matrix. mag[n] = sum_g |dw * dx * S| (binary64), the
 * scale of the terms that the tolerance of a reordered binary32 sum refers to.
 * Every y[n] is computed on its own, so how the columns are split among
 * threads does not change any result. */
static void row_product(const int8_t* qxr, const float* dxr, int64_t n0, int64_t n1, int64_t K,
                        const void* qw, int wbits, const uint16_t* dw,
                        float* yr, double* magr) {
    int64_t G = K / ORC_GROUP;
    for (int64_t n = n0; n < n1; ++n) {
        double acc = 0.0, mag = 0.0;
        for (int64_t g = 0; g < G; ++g) {
            int64_t s = 0;
            for (int i = 0; i < ORC_GROUP; ++i) {
                int64_t k = g * ORC_GROUP + i;
                int wv = (wbits == 8) ? ((const int8_t*)qw)[n * K + k]
                                      : q4_at((const uint8_t*)qw + n * (K / 2), k);
                s += (int64_t)qxr[k] * wv;
            }
            double t = (double)orc_f16_to_f32(dw[n * G + g]) * (double)dxr[g] * (double)s;
            acc += t;
            mag += fabs(t);
        }
        yr[n] = (float)acc;
        if (magr) magr[n] = mag;
    }
}

/* Column chunk of the work split: threads take (row, chunk) items, so a
 * product with one activation row (decode) still uses every core. */
#define ORC_NCHUNK 64

/* Dense GEMM/GEMV: y [M][ldy] (binary32), mag [M][N] (binary64, may be NULL). */
void orc_qgemm(const int8_t* qx, const float* dx, int64_t M, int64_t N, int64_t K,
               const void* qw, int wbits, const uint16_t* dw,
               float* y, int64_t ldy, double* mag) {
    int64_t G = K / ORC_GROUP;
    int64_t chunks = (N + ORC_NCHUNK - 1) / ORC_NCHUNK;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t it = 0; it < M * chunks; ++it) {
        int64_t m = it / chunks, n0 = (it % chunks) * ORC_NCHUNK;
        int64_t n1 = n0 + ORC_NCHUNK < N ? n0 + ORC_NCHUNK : N;
        row_product(qx + m * K, dx + m * G, n0, n1, K, qw, wbits, dw,
                    y + m * ldy, mag ? mag + m * N : NULL);
    }
}

/* Same as orc_qgemm for a listed subset of activation rows: row i of y/mag is
 * activation row rows[i]. Used to check large problems on sampled rows. */
void orc_qgemm_rows(const int8_t* qx, const float* dx, const int64_t* rows, int64_t R,
                    int64_t N, int64_t K, const void* qw, int wbits, const uint16_t* dw,
                    float* y, double* mag) {
    int64_t G = K / ORC_GROUP;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < R; ++i)
        row_product(qx + rows[i] * K, dx + rows[i] * G, 0, N, K, qw, wbits, dw,
                    y + i * N, mag ? mag + i * N : NULL);
}

/* ---- MoE routing and the grouped product ------------------------------------ *
 * Pairs p = token * topk + slot. Routing groups the valid pairs by expert,
 * keeping (token, slot) order inside each expert:
 *   counts[e]   = number of pairs with expert e,
 *   offsets[e]  = sum of counts[0..e-1]  (offsets[E] = number of valid pairs),
 *   perm[...]   = the pair indices, expert by expert.
 * Pairs whose expert id is outside [0, E) are not routed; the return value is
 * how many there were. */
int64_t orc_moe_route(const int32_t* topk_ids, int64_t T, int32_t topk, int32_t E,
                      int32_t* counts, int32_t* offsets, int32_t* perm) {
    int64_t P = T * topk, bad = 0;
    for (int32_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) {
        int32_t e = topk_ids[p];
        if (e < 0 || e >= E) ++bad;
        else ++counts[e];
    }
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int64_t pos = 0;
    for (int32_t e = 0; e < E; ++e)
        for (int64_t p = 0; p < P; ++p)
            if (topk_ids[p] == e) perm[pos++] = (int32_t)p;
    return bad;
}

/* y[p] = x_row(p) * W_{e(p)}^T with Q4_0 expert weights qw4 [E][N][K/2], dw [E][N][G].
 * x_row(p) is activation row p / topk (x_row_mode 0: one row per token) or p
 * (mode 1: one row per pair). Rows of unrouted pairs are zero. Returns the
 * number of unrouted pairs. */
int64_t orc_grouped_qgemm_moe(const int8_t* qx, const float* dx, int64_t K,
                              const int32_t* topk_ids, int64_t T, int32_t topk,
                              int32_t x_row_mode, const uint8_t* qw4, const uint16_t* dw,
                              int32_t E, int64_t N, float* y, double* mag) {
    int64_t P = T * topk, G = K / ORC_GROUP, bad = 0;
    for (int64_t p = 0; p < P; ++p) {
        int32_t e = topk_ids[p];
        if (e < 0 || e >= E) ++bad;
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t p = 0; p < P; ++p) {
        int32_t e = topk_ids[p];
        if (e < 0 || e >= E) {
            for (int64_t n = 0; n < N; ++n) {
                y[p * N + n] = 0.0f;
                if (mag) mag[p * N + n] = 0.0;
            }
            continue;
        }
        int64_t r = x_row_mode ? p : p / topk;
        row_product(qx + r * K, dx + r * G, 0, N, K,
                    qw4 + (int64_t)e * N * (K / 2), 4, dw + (int64_t)e * N * G,
                    y + p * N, mag ? mag + p * N : NULL);
    }
    return bad;
}

/* The MoE steps around the grouped product (readings where the pages are
 * silent: the usual gated expert activation, and a router-weighted sum of
 * the expert rows of each token).
 *
 * h[p][j] = silu(gate) * up with silu(v) = v / (1 + exp(-v)), in binary64,
 * gate = gu[p][j], up = gu[p][F + j]; gu is binary32 [P][ldgu]. */
void orc_silu_mul(const float* gu, int64_t P, int64_t F, int64_t ldgu, double* h) {
    for (int64_t p = 0; p < P; ++p)
        for (int64_t j = 0; j < F; ++j) {
            double g = (double)gu[p * ldgu + j], u = (double)gu[p * ldgu + F + j];
            h[p * F + j] = g / (1.0 + exp(-g)) * u;
        }
}

/* out[t][n] = sum_s w[t][s] * y[t * topk + s][n] in binary64, slot order;
 * mag[t][n] = sum_s |w[t][s] * y[t * topk + s][n]|. */
void orc_moe_combine(const float* y, const float* w, int64_t T, int32_t topk, int64_t N,
                     double* out, double* mag) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, m = 0.0;
            for (int32_t s = 0; s < topk; ++s) {
                double v = (double)w[t * topk + s] * (double)y[(t * topk + s) * N + n];
                acc += v;
                m += fabs(v);
            }
            out[t * N + n] = acc;
            mag[t * N + n] = m;
        }
}

/* GGUF-style interleaved blocks -> planar codes and binary16 scales (the file
 * format the mining-card page's engine reads: per 32 weights a little-endian
 * binary16 scale, then 32 int8 codes (Q8_0) or 16 bytes of nibbles (Q4_0, the
 * same nibble order as the planar qw4)). */
void orc_import_gguf(const uint8_t* blocks, int64_t N, int64_t K, int q4, uint8_t* q,
                     uint16_t* d) {
    int64_t G = K / ORC_GROUP, block_bytes = q4 ? 18 : 34, code_bytes = q4 ? 16 : 32;
    int64_t row_bytes = q4 ? K / 2 : K;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g) {
            const uint8_t* b = blocks + (n * G + g) * block_bytes;
            d[n * G + g] = (uint16_t)(b[0] | (b[1] << 8));
            memcpy(q + n * row_bytes + g * code_bytes, b + 2, (size_t)code_bytes);
        }
}

/* Split-K attention merge in binary64 (the mining-card page, Implementation
 * challenges 3): m = max_s m_s, l = sum_s exp(m_s - m) l_s,
 * o = sum_s exp(m_s - m) acc_s, out = o / l, lse = m + log(l).  Empty splits
 * (m_s = -inf) contribute nothing; an all-empty row gives out = 0, lse = -inf.
 * m, l [S][R], acc [S][R][D]; out [R][D], lse [R], mag [R][D] = sum_s
 * exp(m_s - m) |acc_s| / l (the magnitude a binary32 sum is measured against). */
void orc_splitk_merge(const float* m, const float* l, const float* acc, int32_t S, int64_t R,
                      int64_t D, double* out, double* lse, double* mag) {
    for (int64_t r = 0; r < R; ++r) {
        double mg = -INFINITY;
        for (int32_t s = 0; s < S; ++s)
            if ((double)m[s * R + r] > mg) mg = (double)m[s * R + r];
        double lg = 0.0;
        for (int32_t s = 0; s < S; ++s)
            if (m[s * R + r] != -INFINITY) lg += exp((double)m[s * R + r] - mg) * (double)l[s * R + r];
        lse[r] = lg > 0.0 ? mg + log(lg) : -INFINITY;
        for (int64_t c = 0; c < D; ++c) {
            double o = 0.0, a = 0.0;
            for (int32_t s = 0; s < S; ++s) {
                if (m[s * R + r] == -INFINITY) continue;
                double w = exp((double)m[s * R + r] - mg), v = (double)acc[(s * R + r) * D + c];
                o += w * v;
                a += w * fabs(v);
            }
            out[r * D + c] = lg > 0.0 ? o / lg : 0.0;
            mag[r * D + c] = lg > 0.0 ? a / lg : 0.0;
        }
    }
}

/* 3-bit KV-cache codec (the mining-card page, Features: 3-bit Walsh-Hadamard +
 * Lloyd-Max KV cache; the steps are named only, so the reading is spelled out):
 * codebook: the 8-level Lloyd-Max quantizer of the standard normal law, found
 * by alternating the two optimality conditions (threshold = midpoint of its
 * two levels; level = mean of the law over its cell) in binary64 from evenly
 * spaced starting levels until they stop moving. */
void orc_kv3_codebook(double* levels, double* thresholds) {
    double lv[8], t[9];
    for (int k = 0; k < 8; ++k) lv[k] = -2.0 + 4.0 * k / 7.0;
    for (int it = 0; it < 20000; ++it) {
        t[0] = -INFINITY;
        t[8] = INFINITY;
        for (int k = 1; k < 8; ++k) t[k] = (lv[k - 1] + lv[k]) / 2.0;
        double moved = 0.0;
        for (int k = 0; k < 8; ++k) {
            /* mean of N(0,1) over (a, b): (phi(a) - phi(b)) / (Phi(b) - Phi(a)) */
            double a = t[k], b = t[k + 1];
            double pa = isinf(a) ? 0.0 : exp(-a * a / 2.0) / sqrt(2.0 * acos(-1.0));
            double pb = isinf(b) ? 0.0 : exp(-b * b / 2.0) / sqrt(2.0 * acos(-1.0));
            double Pa = isinf(a) ? 0.0 : 0.5 * erfc(-a / sqrt(2.0));
            double Pb = isinf(b) ? 1.0 : 0.5 * erfc(-b / sqrt(2.0));
            double c = (pa - pb) / (Pb - Pa);
            moved = fmax(moved, fabs(c - lv[k]));
            lv[k] = c;
        }
        if (moved == 0.0) break;
    }
    for (int k = 0; k < 8; ++k) levels[k] = lv[k];
    for (int k = 0; k < 7; ++k) thresholds[k] = (lv[k] + lv[k + 1]) / 2.0;
}

/* Orthonormal Walsh-Hadamard transform of v[0..D) in place (Sylvester order),
 * binary64: pairs (i, i + h) become (v_i + v_{i+h}, v_i - v_{i+h}) for
 * h = 1, 2, .., D/2, then everything is divided by sqrt(D). */
static void wht64(double* v, int D) {
    for (int h = 1; h < D; h *= 2)
        for (int i = 0; i < D; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                double a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
    double r = sqrt((double)D);
    for (int j = 0; j < D; ++j) v[j] /= r;
}

void orc_wht(const double* x, int64_t T, int D, double* y) {
    for (int64_t t = 0; t < T; ++t) {
        memcpy(y + t * D, x + t * D, sizeof(double) * (size_t)D);
        wht64(y + t * D, D);
    }
}

/* Encode: y = H x / sqrt(D) and s = sqrt(mean y^2) in binary64; the stored
 * scale is s rounded to binary32; code = number of binary32 thresholds <= y / s
 * (0 when s == 0), with u = y / s kept for the caller.  Bit planes: word
 * b * (D/32) + e, bit L = bit b of the code of element L * (D/32) + e. */
void orc_kv3_encode(const float* x, int64_t T, int D, const float* thr32, uint32_t* codes,
                    float* scales, double* u_out) {
    int E = D / 32;
    double y[256];
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < D; ++j) y[j] = (double)x[t * D + j];
        wht64(y, D);
        double ss = 0.0;
        for (int j = 0; j < D; ++j) ss += y[j] * y[j];
        double s = sqrt(ss / D);
        scales[t] = (float)s;
        uint32_t* w = codes + t * 3 * E;
        for (int i = 0; i < 3 * E; ++i) w[i] = 0;
        for (int j = 0; j < D; ++j) {
            double u = s > 0.0 ? y[j] / s : 0.0;
            int k = 0;
            if (s > 0.0)
                for (int i = 0; i < 7; ++i) k += u >= (double)thr32[i];
            u_out[t * D + j] = u;
            int L = j / E, e = j % E;
            for (int b = 0; b < 3; ++b)
                if ((k >> b) & 1) w[b * E + e] |= 1u << L;
        }
    }
}

/* Decode: y^_j = s * level[code_j] (binary32 levels), x^ = H y^ / sqrt(D), binary64. */
void orc_kv3_decode(const uint32_t* codes, const float* scales, int64_t T, int D,
                    const float* lv32, double* out) {
    int E = D / 32;
    for (int64_t t = 0; t < T; ++t) {
        const uint32_t* w = codes + t * 3 * E;
        double* y = out + t * D;
        for (int j = 0; j < D; ++j) {
            int L = j / E, e = j % E, k = 0;
            for (int b = 0; b < 3; ++b) k |= (int)((w[b * E + e] >> L) & 1u) << b;
            y[j] = (double)scales[t] * (double)lv32[k];
        }
        wht64(y, D);
    }
}
