/*
 * ORACLE for MoE token dispatch + expert GEMM. TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library. It shares no code with the CUDA path: no headers, no
 * helpers, no tables. It is deliberately plain and slow: serial loops in the
 * order the definitions are written, floating point in float64.
 *
 * What it computes (the expert-parallel "token-dispatch + GEMM" of
 * "Loads and Loads of Fluffy Kittens", section "Key claims", Fig. 17, on one
 * device): given routed expert indices topk[T][k],
 *   1. count[e]   = number of (t, s) with topk[t][s] == e;
 *   2. offsets[0] = 0, offsets[e+1] = offsets[e] + count[e];
 *   3. perm       = the flat routing indices f = t*k + s listed expert by
 *                   expert, and inside one expert by increasing f (token,
 *                   then slot); inv_perm[f] = position of f in perm;
 *   4. out[j][n]  = sum over d of x[perm[j] / k][d] * W[e(j)][d][n], where
 *                   e(j) is the expert whose segment [offsets[e],
 *                   offsets[e+1]) holds j. Inputs are bf16, the products
 *                   and the sum are formed in float64, d ascending.
 *
 * All integer outputs are int64 so that nothing about their width is shared
 * with the device path (which uses int32).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bit pattern -> float64; exact (bf16 is the top half of a float32). */
double oracle_bf16_to_f64(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Step 1 and 2. Returns 0, or 1 if an index is outside [0, E). */
int oracle_route_counts(const int32_t* topk, int64_t T, int64_t k, int64_t E,
                        int64_t* counts, int64_t* offsets) {
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t s = 0; s < k; ++s) {
            int64_t e = topk[t * k + s];
            if (e < 0 || e >= E) return 1;
            counts[e] += 1;
        }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    return 0;
}

/* Step 3: counting-sort scatter, visiting (t, s) in increasing order, so the
 * order inside each expert's segment is the visiting order (stable). */
int oracle_build_perm(const int32_t* topk, int64_t T, int64_t k, int64_t E,
                      const int64_t* offsets, int64_t* perm, int64_t* inv_perm) {
    int64_t* cursor = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
    if (!cursor) return 2;
    for (int64_t e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t t = 0; t < T; ++t)
        for (int64_t s = 0; s < k; ++s) {
            int64_t f = t * k + s;
            int64_t e = topk[f];
            if (e < 0 || e >= E) { free(cursor); return 1; }
            int64_t j = cursor[e]++;
            perm[j] = f;
            if (inv_perm) inv_perm[f] = j;
        }
    free(cursor);
    return 0;
}

/* e(j): the expert whose segment holds row j (empty segments hold nothing). */
int64_t oracle_expert_of_row(const int64_t* offsets, int64_t E, int64_t j) {
    for (int64_t e = 0; e < E; ++e)
        if (offsets[e] <= j && j < offsets[e + 1]) return e;
    return -1;
}

/* Step 4 for one row j: out[n] for n in [0, De). */
static int gemm_one_row(const uint16_t* x, const int64_t* perm, const int64_t* offsets,
                        const uint16_t* W, int64_t T, int64_t k, int64_t D, int64_t E,
                        int64_t De, int64_t j, double* out) {
    int64_t e = oracle_expert_of_row(offsets, E, j);
    if (e < 0) return 1;
    int64_t t = perm[j] / k;
    if (t < 0 || t >= T) return 1;
    for (int64_t n = 0; n < De; ++n) out[n] = 0.0;
    for (int64_t d = 0; d < D; ++d) {
        double xv = oracle_bf16_to_f64(x[t * D + d]);
        const uint16_t* wrow = W + ((size_t)e * (size_t)D + (size_t)d) * (size_t)De;
        for (int64_t n = 0; n < De; ++n) out[n] += xv * oracle_bf16_to_f64(wrow[n]);
    }
    return 0;
}

typedef struct {
    const uint16_t *x, *W;
    const int64_t *perm, *offsets, *rows;
    int64_t T, k, D, E, De, r0, r1;
    double* out;
    int status;
} gemm_job;

static void* gemm_worker(void* arg) {
    gemm_job* g = (gemm_job*)arg;
    g->status = 0;
    for (int64_t r = g->r0; r < g->r1; ++r)
        if (gemm_one_row(g->x, g->perm, g->offsets, g->W, g->T, g->k, g->D, g->E, g->De,
                         g->rows[r], g->out + (size_t)r * (size_t)g->De))
            g->status = 1;
    return NULL;
}

/* Step 4 for the listed rows: out[r][n] = result for row rows[r].
 * Threads split the list of rows; each row is computed by one thread in the
 * serial order above, so the result does not depend on nthreads. */
int oracle_gemm_rows(const uint16_t* x, const int64_t* perm, const int64_t* offsets,
                     const uint16_t* W, int64_t T, int64_t k, int64_t D, int64_t E, int64_t De,
                     const int64_t* rows, int64_t nrows, double* out, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
    pthread_t th[256];
    gemm_job jobs[256];
    int created[256];
    int64_t per = (nrows + nthreads - 1) / nthreads;
    int n = 0;
    for (int i = 0; i < nthreads; ++i) {
        int64_t b = i * per, e = b + per;
        if (b >= nrows) break;
        if (e > nrows) e = nrows;
        gemm_job g = {x, W, perm, offsets, rows, T, k, D, E, De, b, e, out, 0};
        jobs[i] = g;
        created[i] = (i < nthreads - 1) && pthread_create(&th[i], NULL, gemm_worker, &jobs[i]) == 0;
        if (!created[i]) gemm_worker(&jobs[i]);
        n = i + 1;
    }
    int status = 0;
    for (int i = 0; i < n; ++i) {
        if (created[i]) pthread_join(th[i], NULL);
        status |= jobs[i].status;
    }
    return status;
}

/* ---------------------------------------------------------------------- */
/* Combine (un-permute and weight) -- the step after the expert MLP in the
 * expert-parallel token-dispatch + GEMM of "Loads and Loads of Fluffy
 * Kittens" ("Key claims", Fig. 17), whose gating the pages leave open:
 *   y[t][c] = sum over s = 0..k-1 of gates[t][s] * src[inv_perm[t*k + s]][c]
 * with src in bf16 and the products and sum in float64, s ascending.
 * Returns 0, or 1 if an inv_perm entry is outside [0, T*k). */
int oracle_combine(const uint16_t* src, const int64_t* inv_perm, const double* gates, int64_t T,
                   int64_t k, int64_t C, double* y) {
    const int64_t R = T * k;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < C; ++c) y[t * C + c] = 0.0;
        for (int64_t s = 0; s < k; ++s) {
            const int64_t j = inv_perm[t * k + s];
            if (j < 0 || j >= R) return 1;
            const double g = gates[t * k + s];
            for (int64_t c = 0; c < C; ++c)
                y[t * C + c] += g * oracle_bf16_to_f64(src[j * C + c]);
        }
    }
    return 0;
}

/* Router top-k: for every token t, the k experts with the largest logits,
 * largest first, equal logits going to the lower expert index; and gates =
 * softmax over the k selected logits (float64, shifted by the largest).
 * The pages fix top_k and num_experts ("Key claims", Fig. 17) but not the
 * router; this is the plainest reading. */
int oracle_router_topk(const float* logits, int64_t T, int64_t E, int64_t k, int64_t* topk,
                       double* gates) {
    if (k < 1 || k > E) return 1;
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!taken) return 2;
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        for (int64_t e = 0; e < E; ++e) taken[e] = 0;
        for (int64_t s = 0; s < k; ++s) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            topk[t * k + s] = best;
        }
        const double m = (double)l[topk[t * k]];
        double z = 0.0;
        for (int64_t s = 0; s < k; ++s) z += exp((double)l[topk[t * k + s]] - m);
        for (int64_t s = 0; s < k; ++s) gates[t * k + s] = exp((double)l[topk[t * k + s]] - m) / z;
    }
    free(taken);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* FP8 (E4M3) weights and activations: the "FP8 weights" variant of the
 * expert GEMM (the pages mention FP8 tensor-core support for Blackwell only
 * in passing; the quantisation scheme here is a reading). Codes follow the
 * OCP 8-bit floating point E4M3 format: 1 sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits, largest finite 448, no infinities, NaN = S.1111.111.
 * Conversion: round to nearest, ties to even; magnitudes above 448 saturate
 * to 448 (as the hardware's satfinite conversion does). */
uint8_t oracle_f32_to_e4m3(float f) {
    const uint8_t sign = signbit(f) ? 0x80u : 0u;
    if (isnan(f)) return (uint8_t)(sign | 0x7Fu);
    const double a = fabs((double)f);
    if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
    if (a < 0.015625) { /* below the smallest normal 2^-6: steps of 2^-9 */
        const double m = rint(a * 512.0); /* 0..8; 8 is the smallest normal */
        return (uint8_t)(sign | (uint8_t)m);
    }
    int e = (int)floor(log2(a));
    if (ldexp(1.0, e) > a) e -= 1;          /* guard log2 rounding */
    if (ldexp(1.0, e + 1) <= a) e += 1;
    double m = rint((a / ldexp(1.0, e) - 1.0) * 8.0); /* 0..8 */
    if (m >= 8.0) { m = 0.0; e += 1; }
    uint32_t code = (uint32_t)((e + 7) << 3) | (uint32_t)m;
    if (code > 0x7Eu) code = 0x7Eu;
    return (uint8_t)(sign | code);
}

double oracle_e4m3_to_f64(uint8_t c) {
    const double s = (c & 0x80u) ? -1.0 : 1.0;
    const int e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) return s * ldexp((double)m, -9);
    return s * ldexp(1.0 + m / 8.0, e - 7);
}

/* One vector quantised with one scale, in float32 arithmetic:
 *   amax = max |v|,  inv = 448 / amax,  code = E4M3(v * inv),
 *   scale = amax / 448.
 * When amax == 0, or amax is so small (below 448 / FLT_MAX, about 1.3e-36)
 * that 448 / amax overflows, inv = scale = 1: every |v| is then far below
 * E4M3's smallest step and every code is zero, as for an all-zero vector.
 * Inputs are finite. */
static void quant_vec(const uint16_t* v, int64_t n, int64_t stride, uint8_t* q, int64_t qstride,
                      float* scale) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float a = fabsf((float)oracle_bf16_to_f64(v[i * stride]));
        if (a > amax) amax = a;
    }
    const float r = 448.0f / amax;
    const int plain = amax > 0.0f && isfinite(r);
    const float inv = plain ? r : 1.0f;
    *scale = plain ? amax / 448.0f : 1.0f;
    for (int64_t i = 0; i < n; ++i)
        q[i * qstride] = oracle_f32_to_e4m3((float)oracle_bf16_to_f64(v[i * stride]) * inv);
}

/* Rows of x [T, D]: xq [T, D], sx [T]. */
void oracle_quant_rows(const uint16_t* x, int64_t T, int64_t D, uint8_t* xq, float* sx) {
    for (int64_t t = 0; t < T; ++t) quant_vec(x + t * D, D, 1, xq + t * D, 1, sx + t);
}

/* Columns of every W[e] [D, N]: codes stored transposed, wq [E, N, D] (each
 * output column's D codes contiguous), sw [E, N]. */
void oracle_quant_cols(const uint16_t* W, int64_t E, int64_t D, int64_t N, uint8_t* wq,
                       float* sw) {
    for (int64_t e = 0; e < E; ++e)
        for (int64_t n = 0; n < N; ++n)
            quant_vec(W + e * D * N + n, D, N, wq + (e * N + n) * D, 1, sw + e * N + n);
}

/* The FP8 expert GEMM for the listed sorted rows, float64 from the codes:
 *   out[j][n] = (sum_d q(x)[t][d] * q(W)[e][n][d]) * sx[t] * sw[e][n],
 * t = perm[j] / k, e = e(j). */
int oracle_gemm_fp8_rows(const uint8_t* xq, const float* sx, const int64_t* perm,
                         const int64_t* offsets, const uint8_t* wq, const float* sw, int64_t T,
                         int64_t k, int64_t D, int64_t E, int64_t N, const int64_t* rows,
                         int64_t nrows, double* out) {
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t j = rows[r];
        const int64_t e = oracle_expert_of_row(offsets, E, j);
        if (e < 0) return 1;
        const int64_t t = perm[j] / k;
        if (t < 0 || t >= T) return 1;
        for (int64_t n = 0; n < N; ++n) {
            const uint8_t* wcol = wq + (e * N + n) * D;
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d)
                acc += oracle_e4m3_to_f64(xq[t * D + d]) * oracle_e4m3_to_f64(wcol[d]);
            out[r * N + n] = acc * (double)sx[t] * (double)sw[e * N + n];
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Microscaling FP8 (MXFP8), the block-scaled FP8 form that the tutorial
 * page's "ThunderKittens 2.0 & FP8/NVFP4" item names. The pages do not
 * define it; this follows the definition of the MX formats (OCP Microscaling
 * Formats specification): 32 consecutive elements along the reduction
 * dimension share one scale X = 2^s, stored as an 8-bit power of two (E8M0:
 * the byte s + 127), and each element is the E4M3 code of v / X. One block:
 *   amax = max |v_i|;
 *   s    = floor(log2(amax)) - 8, clamped to [-127, 127] (8 is the exponent
 *          of E4M3's largest normal value, 448 = 1.75 * 2^8), so that the
 *          block's largest magnitude lands in [256, 512) before conversion;
 *   code_i = E4M3(v_i / 2^s): round to nearest even, magnitudes above 448
 *          saturated to 448 (only the block maximum can reach [448, 512));
 *   an all-zero block takes s = -127 (byte 0) and zero codes.
 * The dequantised element is value(code_i) * 2^s; v / 2^s is formed exactly
 * (a power-of-two scaling of a bf16 value). */
static int mx_shared_exp(double amax) {
    if (amax == 0.0) return -127;
    int e = (int)floor(log2(amax));
    if (ldexp(1.0, e) > amax) e -= 1;      /* guard log2 rounding */
    if (ldexp(1.0, e + 1) <= amax) e += 1;
    int s = e - 8;
    if (s < -127) s = -127;
    if (s > 127) s = 127;
    return s;
}

/* One block of n values `stride` apart -> n codes `qstride` apart; returns
 * the E8M0 byte. */
static uint8_t mx_block(const uint16_t* v, int64_t n, int64_t stride, uint8_t* q, int64_t qstride) {
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double a = fabs(oracle_bf16_to_f64(v[i * stride]));
        if (a > amax) amax = a;
    }
    const int s = mx_shared_exp(amax);
    for (int64_t i = 0; i < n; ++i)
        q[i * qstride] = oracle_f32_to_e4m3((float)ldexp(oracle_bf16_to_f64(v[i * stride]), -s));
    return (uint8_t)(s + 127);
}

/* E8M0 byte -> its power of two (byte 255 is NaN in the format; unused here). */
double oracle_e8m0_to_f64(uint8_t b) {
    if (b == 255u) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* Rows of x [T, D], D a multiple of 32: xq [T, D] codes, sx [T, D / 32]
 * E8M0 bytes (block b of row t covers d in [32 b, 32 b + 32)). Returns 1 if
 * D is not a multiple of 32. */
int oracle_mx_quant_rows(const uint16_t* x, int64_t T, int64_t D, uint8_t* xq, uint8_t* sx) {
    if (D % 32 != 0) return 1;
    const int64_t nb = D / 32;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t b = 0; b < nb; ++b)
            sx[t * nb + b] = mx_block(x + t * D + 32 * b, 32, 1, xq + t * D + 32 * b, 1);
    return 0;
}

/* Columns of every W[e] [D, N] (blocks along d): codes stored transposed,
 * wq [E, N, D] (each output column's D codes contiguous), sw [E, N, D / 32].
 * Returns 1 if D is not a multiple of 32. */
int oracle_mx_quant_cols(const uint16_t* W, int64_t E, int64_t D, int64_t N, uint8_t* wq,
                         uint8_t* sw) {
    if (D % 32 != 0) return 1;
    const int64_t nb = D / 32;
    for (int64_t e = 0; e < E; ++e)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < nb; ++b)
                sw[(e * N + n) * nb + b] = mx_block(W + (e * D + 32 * b) * N + n, 32, N,
                                                    wq + (e * N + n) * D + 32 * b, 1);
    return 0;
}

/* The MXFP8 expert GEMM for the listed sorted rows, float64:
 *   out[j][n] = sum_d (value(xq[t][d]) * 2^(sx[t][d/32] - 127))
 *                   * (value(wq[e][n][d]) * 2^(sw[e][n][d/32] - 127)),
 * d ascending, t = perm[j] / k, e = e(j). */
int oracle_gemm_mx_rows(const uint8_t* xq, const uint8_t* sx, const int64_t* perm,
                        const int64_t* offsets, const uint8_t* wq, const uint8_t* sw, int64_t T,
                        int64_t k, int64_t D, int64_t E, int64_t N, const int64_t* rows,
                        int64_t nrows, double* out) {
    if (D % 32 != 0) return 1;
    const int64_t nb = D / 32;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t j = rows[r];
        const int64_t e = oracle_expert_of_row(offsets, E, j);
        if (e < 0) return 1;
        const int64_t t = perm[j] / k;
        if (t < 0 || t >= T) return 1;
        for (int64_t n = 0; n < N; ++n) {
            const uint8_t* wcol = wq + (e * N + n) * D;
            const uint8_t* wsc = sw + (e * N + n) * nb;
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d)
                acc += (oracle_e4m3_to_f64(xq[t * D + d]) * oracle_e8m0_to_f64(sx[t * nb + d / 32])) *
                       (oracle_e4m3_to_f64(wcol[d]) * oracle_e8m0_to_f64(wsc[d / 32]));
            out[r * N + n] = acc;
        }
    }
    return 0;
}
