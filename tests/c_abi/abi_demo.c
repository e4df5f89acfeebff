/* The C ABI used from plain C (no Python, no torch): device buffers from
 * cudaMalloc, the three calls of the path on a CUDA stream, and the result
 * checked against the CPU oracle (a separate library; test infrastructure).
 * Exit status 0 when counts, offsets, perm and inv_perm match bit for bit
 * and every GEMM output is within |gpu - ref| <= 2e-2 + 1e-2 |ref|. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "pk_moe.h"

/* seeded input generator (inputgen/gen.c) */
int ig_fill_normal_bf16(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n, double scale,
                        uint16_t* out, int nthreads);
int ig_topk_routing(uint64_t seed, uint64_t stream, int64_t T, int64_t E, int64_t k,
                    double zipf_s, int32_t* topk, int nthreads);
/* oracle (oracle/oracle.c) */
int oracle_route_counts(const int32_t* topk, int64_t T, int64_t k, int64_t E, int64_t* counts,
                        int64_t* offsets);
int oracle_build_perm(const int32_t* topk, int64_t T, int64_t k, int64_t E,
                      const int64_t* offsets, int64_t* perm, int64_t* inv_perm);
int oracle_gemm_rows(const uint16_t* x, const int64_t* perm, const int64_t* offsets,
                     const uint16_t* W, int64_t T, int64_t k, int64_t D, int64_t E, int64_t De,
                     const int64_t* rows, int64_t nrows, double* out, int nthreads);

#define CHECK_CUDA(call)                                                            \
    do {                                                                            \
        cudaError_t e_ = (call);                                                    \
        if (e_ != cudaSuccess) {                                                    \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));             \
            return 2;                                                               \
        }                                                                           \
    } while (0)
#define CHECK_PK(call)                                                              \
    do {                                                                            \
        int r_ = (call);                                                            \
        if (r_ != PK_OK) {                                                          \
            fprintf(stderr, "%s: %s\n", #call, pk_status_str(r_));                  \
            return 3;                                                               \
        }                                                                           \
    } while (0)

static double bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int main(void) {
    /* several m-tiles and a ragged n-tile: 2048 routed rows over 16 experts */
    const int32_t T = 512, D = 576, E = 16, k = 4, De = 320;
    const int64_t R = (int64_t)T * k;
    uint16_t* x = malloc(sizeof(uint16_t) * T * D);
    uint16_t* W = malloc(sizeof(uint16_t) * E * D * De);
    int32_t* topk = malloc(sizeof(int32_t) * R);
    if (!x || !W || !topk) return 4;
    if (ig_fill_normal_bf16(0, 1, 0, (uint64_t)T * D, 1.0, x, 4) ||
        ig_fill_normal_bf16(0, 2, 0, (uint64_t)E * D * De, 1.0 / sqrt((double)D), W, 4) ||
        ig_topk_routing(0, 3, T, E, k, 0.0, topk, 4))
        return 4;

    uint16_t *dx, *dW, *dout;
    int32_t *dtopk, *dcounts, *doffsets, *dperm, *dinv, *dstatus;
    void* dws;
    const size_t ws = pk_moe_workspace_bytes(T, k, E);
    CHECK_CUDA(cudaMalloc((void**)&dx, sizeof(uint16_t) * T * D));
    CHECK_CUDA(cudaMalloc((void**)&dW, sizeof(uint16_t) * E * D * De));
    CHECK_CUDA(cudaMalloc((void**)&dout, sizeof(uint16_t) * R * De));
    CHECK_CUDA(cudaMalloc((void**)&dtopk, sizeof(int32_t) * R));
    CHECK_CUDA(cudaMalloc((void**)&dcounts, sizeof(int32_t) * E));
    CHECK_CUDA(cudaMalloc((void**)&doffsets, sizeof(int32_t) * (E + 1)));
    CHECK_CUDA(cudaMalloc((void**)&dperm, sizeof(int32_t) * R));
    CHECK_CUDA(cudaMalloc((void**)&dinv, sizeof(int32_t) * R));
    CHECK_CUDA(cudaMalloc((void**)&dstatus, sizeof(int32_t)));
    CHECK_CUDA(cudaMalloc(&dws, ws > 0 ? ws : 16));
    CHECK_CUDA(cudaMemcpy(dx, x, sizeof(uint16_t) * T * D, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dW, W, sizeof(uint16_t) * E * D * De, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dtopk, topk, sizeof(int32_t) * R, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemset(dstatus, 0, sizeof(int32_t)));

    cudaStream_t s;
    CHECK_CUDA(cudaStreamCreate(&s));
    CHECK_PK(pk_moe_route_counts(dtopk, T, k, E, dcounts, doffsets, dws, ws, dstatus, s));
    CHECK_PK(pk_moe_build_perm(dtopk, T, k, E, doffsets, dperm, dinv, dws, ws, dstatus, s));
    CHECK_PK(pk_moe_dispatch_gemm(dx, dperm, doffsets, dW, T, k, D, E, De, dout, dstatus, s));
    CHECK_CUDA(cudaStreamSynchronize(s));

    int32_t status = -1;
    int32_t* counts = malloc(sizeof(int32_t) * E);
    int32_t* offsets = malloc(sizeof(int32_t) * (E + 1));
    int32_t* perm = malloc(sizeof(int32_t) * R);
    int32_t* inv = malloc(sizeof(int32_t) * R);
    uint16_t* out = malloc(sizeof(uint16_t) * R * De);
    if (!counts || !offsets || !perm || !inv || !out) return 4;
    CHECK_CUDA(cudaMemcpy(&status, dstatus, sizeof status, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(counts, dcounts, sizeof(int32_t) * E, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(offsets, doffsets, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(perm, dperm, sizeof(int32_t) * R, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(inv, dinv, sizeof(int32_t) * R, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(out, dout, sizeof(uint16_t) * R * De, cudaMemcpyDeviceToHost));
    if (status != PK_OK) {
        fprintf(stderr, "device status: %s\n", pk_status_str(status));
        return 5;
    }

    int64_t* rcounts = malloc(sizeof(int64_t) * E);
    int64_t* roffsets = malloc(sizeof(int64_t) * (E + 1));
    int64_t* rperm = malloc(sizeof(int64_t) * R);
    int64_t* rinv = malloc(sizeof(int64_t) * R);
    int64_t* rows = malloc(sizeof(int64_t) * R);
    double* ref = malloc(sizeof(double) * R * De);
    if (!rcounts || !roffsets || !rperm || !rinv || !rows || !ref) return 4;
    if (oracle_route_counts(topk, T, k, E, rcounts, roffsets) ||
        oracle_build_perm(topk, T, k, E, roffsets, rperm, rinv))
        return 6;
    for (int32_t e = 0; e < E; ++e)
        if (counts[e] != rcounts[e]) return fprintf(stderr, "counts[%d]\n", e), 7;
    for (int32_t e = 0; e <= E; ++e)
        if (offsets[e] != roffsets[e]) return fprintf(stderr, "offsets[%d]\n", e), 7;
    for (int64_t j = 0; j < R; ++j) {
        if (perm[j] != rperm[j]) return fprintf(stderr, "perm[%lld]\n", (long long)j), 7;
        if (inv[j] != rinv[j]) return fprintf(stderr, "inv_perm[%lld]\n", (long long)j), 7;
        rows[j] = j;
    }
    if (oracle_gemm_rows(x, rperm, roffsets, W, T, k, D, E, De, rows, R, ref, 4)) return 6;
    double maxerr = 0.0;
    for (int64_t i = 0; i < R * De; ++i) {
        const double g = bf16_to_double(out[i]), r = ref[i], err = fabs(g - r);
        if (!(err <= 2e-2 + 1e-2 * fabs(r))) {
            fprintf(stderr, "out[%lld]: gpu %g oracle %g\n", (long long)i, g, r);
            return 8;
        }
        if (err > maxerr) maxerr = err;
    }
    printf("c abi demo ok: T=%d D=%d E=%d k=%d D_expert=%d, max |gpu-ref| = %.3g\n", T, D, E, k,
           De, maxerr);
    cudaStreamDestroy(s);
    return 0;
}
