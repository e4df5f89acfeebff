// Host-side declarations shared by the translation units of libpkmoe.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pk_moe.h"

namespace pk {

// Routing: entries of topk_idx (flattened, t*k + s) handled by one block.
constexpr int kRouteChunk = 2048;
constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;

inline int route_blocks(int64_t R) { return static_cast<int>((R + kRouteChunk - 1) / kRouteChunk); }

cudaError_t launch_route_counts(const int32_t* topk, int32_t R, int32_t E, int32_t* counts,
                                int32_t* offsets, int32_t* blockbase, int32_t* status,
                                cudaStream_t stream);
// Kernels launched by launch_route_counts + launch_build_perm for R entries.
int route_kernel_launches(int64_t R, int32_t E);
cudaError_t launch_build_perm(const int32_t* topk, int32_t R, int32_t E,
                              const int32_t* blockbase, int32_t* perm, int32_t* inv_perm,
                              int32_t* status, cudaStream_t stream);

// Dispatch GEMM, one-CTA kernel. Returns PK_OK or a pk_status for host-side
// failures.
int launch_dispatch_gemm_single(const uint16_t* x, const int32_t* perm, const int32_t* offsets,
                         const uint16_t* W, int32_t T, int32_t k, int32_t D, int32_t E,
                         int32_t De, uint16_t* out, int32_t* status, cudaStream_t stream,
                         uint64_t wait_limit_ns);

// FP8 dispatch GEMM: E4M3 codes xq [T, D] and wq [E, De, D] with fp32 scales
// sx [T] and sw [E, De].
int launch_dispatch_gemm_fp8_single(const uint8_t* xq, const float* sx, const int32_t* perm,
                             const int32_t* offsets, const uint8_t* wq, const float* sw,
                             int32_t T, int32_t k, int32_t D, int32_t E, int32_t De,
                             uint16_t* out, int32_t* status, cudaStream_t stream,
                             uint64_t wait_limit_ns);

// Dispatch GEMM on CTA pairs (bf16, or FP8 codes with scales sx, sw).
int launch_dispatch_gemm_pair(bool fp8, const void* x, const float* sx, const int32_t* perm,
                              const int32_t* offsets, const void* W, const float* sw, int32_t T,
                              int32_t k, int32_t D, int32_t E, int32_t De, uint16_t* out,
                              int32_t* status, cudaStream_t stream, uint64_t wait_limit_ns);

// Tensor map of bf16 W [E, D, De] or of the blocked FP8 codes.
int make_w_map(bool fp8, const void* W, int32_t D, int32_t E, int32_t De, CUtensorMap* wmap);

// E4M3 quantisation with one scale per row of x / per (expert, column) of W.
cudaError_t launch_quant_rows(const uint16_t* x, int32_t T, int32_t D, uint8_t* q, float* scale,
                              cudaStream_t stream);
cudaError_t launch_quant_cols(const uint16_t* W, int32_t E, int32_t D, int32_t N, uint8_t* q,
                              float* scale, cudaStream_t stream);

// FP8 grouped GEMM: E4M3 codes Aq [R, K] (scales sa [R]) and blocked W codes
// (scales sw [E, N]).
int launch_grouped_gemm_fp8(const uint8_t* Aq, const float* sa, const int32_t* offsets,
                            const uint8_t* wq, const float* sw, int32_t R, int32_t K, int32_t N,
                            int32_t E, uint16_t* out, int32_t* status, cudaStream_t stream,
                            uint64_t wait_limit_ns);

// Grouped GEMM of expert-sorted rows (no gather).
int launch_grouped_gemm(const uint16_t* A, const int32_t* offsets, const uint16_t* W, int32_t R,
                        int32_t K, int32_t N, int32_t E, uint16_t* out, int32_t* status,
                        cudaStream_t stream, uint64_t wait_limit_ns);

// MXFP8: E4M3 codes with one E8M0 scale byte per 32 elements along D.
// Rows of x: codes [T, D], scales [T, D / 32]. Weights: codes in the FP8
// blocked layout, scales in the blocked layout of the MX GEMM (D % 128 == 0).
size_t mx_weight_scale_bytes(int32_t E, int32_t D, int32_t N);
cudaError_t launch_quant_rows_mx(const uint16_t* x, int32_t T, int32_t D, uint8_t* q, uint8_t* s,
                                 cudaStream_t stream);
cudaError_t launch_quant_cols_mx(const uint16_t* W, int32_t E, int32_t D, int32_t N, uint8_t* q,
                                 uint8_t* sb, cudaStream_t stream);
// MXFP8 dispatch GEMM (block-scaled tensor-core MMAs).
int launch_dispatch_gemm_mx(const uint8_t* xq, const uint8_t* sx, const int32_t* perm,
                            const int32_t* offsets, const uint8_t* wq, const uint8_t* swb,
                            int32_t T, int32_t k, int32_t D, int32_t E, int32_t De, uint16_t* out,
                            int32_t* status, cudaStream_t stream, uint64_t wait_limit_ns);

cudaError_t launch_bounded_wait_probe(int32_t* status, uint64_t limit_ns, cudaStream_t stream);
// Test hook of the one-CTA GEMM kernels: CTA `cta` skips the copies of its
// K-step `kstep` (counted over its units); cta < 0 turns it off.
void set_debug_stall(int32_t cta, int64_t kstep);

cudaError_t launch_router_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                               int32_t* topk, float* gates, cudaStream_t stream);
cudaError_t launch_combine(const uint16_t* src, const int32_t* inv_perm, const float* gates,
                           int32_t T, int32_t k, int32_t C, uint16_t* y, int32_t* status,
                           cudaStream_t stream);

}  // namespace pk
