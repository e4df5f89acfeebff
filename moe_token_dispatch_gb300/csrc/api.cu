// extern "C" entry points of libpkmoe.so: argument checks, then launches.
// Every check that can fail runs before any CUDA call, so a rejected call
// touches neither the device nor the stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pk_internal.h"

namespace {

constexpr uint64_t kDefaultWaitLimitNs = 4000000000ull;
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int> g_gemm_kernel{PK_GEMM_KERNEL_AUTO};

// The one-CTA kernel is the default: on GB300 it is faster on every measured
// workload (the pair kernel pays a cross-SM handshake on every K-step).
bool use_pair() {
    return g_gemm_kernel.load(std::memory_order_relaxed) == PK_GEMM_KERNEL_PAIR;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

const char* pk_status_str(int status) {
    switch (status) {
        case PK_OK: return "PK_OK";
        case PK_ERR_INVALID_ARG: return "PK_ERR_INVALID_ARG";
        case PK_ERR_UNSUPPORTED: return "PK_ERR_UNSUPPORTED";
        case PK_ERR_CUDA: return "PK_ERR_CUDA";
        case PK_ERR_TIMEOUT: return "PK_ERR_TIMEOUT";
        case PK_ERR_BAD_INDEX: return "PK_ERR_BAD_INDEX";
        case PK_ERR_CAPTURE: return "PK_ERR_CAPTURE";
        default: return "PK_ERR_UNKNOWN";
    }
}

int pk_abi_version(void) { return PK_ABI_VERSION; }

size_t pk_moe_workspace_bytes(int32_t T, int32_t k, int32_t E) {
    if (T <= 0 || k <= 0 || E <= 0) return 0;
    const int64_t R = static_cast<int64_t>(T) * k;
    const size_t bytes = static_cast<size_t>(pk::route_blocks(R)) * static_cast<size_t>(E) * 4u;
    return (bytes + 255u) & ~static_cast<size_t>(255u);
}

int pk_moe_route_counts(const int32_t* topk_idx, int32_t T, int32_t k, int32_t E,
                        int32_t* expert_counts, int32_t* expert_offsets, void* workspace,
                        size_t workspace_bytes, int32_t* status_word, void* stream) {
    if (T < 0 || k < 1 || E < 1 || k > E || !expert_offsets) return PK_ERR_INVALID_ARG;
    if (E > PK_MAX_EXPERTS) return PK_ERR_UNSUPPORTED;
    const int64_t R = static_cast<int64_t>(T) * k;
    if (R >= (int64_t{1} << 31)) return PK_ERR_UNSUPPORTED;
    if (R > 0 && (!topk_idx || !workspace)) return PK_ERR_INVALID_ARG;
    if (workspace_bytes < pk_moe_workspace_bytes(T, k, E)) return PK_ERR_INVALID_ARG;
    if (workspace && !aligned16(workspace)) return PK_ERR_INVALID_ARG;
    cudaError_t err = pk::launch_route_counts(topk_idx, static_cast<int32_t>(R), E, expert_counts,
                                              expert_offsets, static_cast<int32_t*>(workspace),
                                              status_word, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

int pk_moe_build_perm(const int32_t* topk_idx, int32_t T, int32_t k, int32_t E,
                      const int32_t* expert_offsets, int32_t* perm, int32_t* inv_perm,
                      const void* workspace, size_t workspace_bytes, int32_t* status_word,
                      void* stream) {
    if (T < 0 || k < 1 || E < 1 || k > E) return PK_ERR_INVALID_ARG;
    if (E > PK_MAX_EXPERTS) return PK_ERR_UNSUPPORTED;
    const int64_t R = static_cast<int64_t>(T) * k;
    if (R >= (int64_t{1} << 31)) return PK_ERR_UNSUPPORTED;
    if (R == 0) return PK_OK;
    if (!topk_idx || !expert_offsets || !perm || !workspace) return PK_ERR_INVALID_ARG;
    if (workspace_bytes < pk_moe_workspace_bytes(T, k, E) || !aligned16(workspace))
        return PK_ERR_INVALID_ARG;
    cudaError_t err = pk::launch_build_perm(topk_idx, static_cast<int32_t>(R), E,
                                            static_cast<const int32_t*>(workspace), perm, inv_perm,
                                            status_word, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

int pk_moe_dispatch_gemm(const uint16_t* x, const int32_t* perm, const int32_t* expert_offsets,
                         const uint16_t* W, int32_t T, int32_t k, int32_t D, int32_t E,
                         int32_t D_expert, uint16_t* out, int32_t* status_word, void* stream) {
    if (T < 0 || k < 1 || E < 1 || D < 1 || D_expert < 1) return PK_ERR_INVALID_ARG;
    if ((D % 8) != 0 || (D_expert % 8) != 0) return PK_ERR_INVALID_ARG;
    const int64_t R = static_cast<int64_t>(T) * k;
    if (R >= (int64_t{1} << 31)) return PK_ERR_UNSUPPORTED;
    if (R == 0) return PK_OK;
    if (!x || !perm || !expert_offsets || !W || !out) return PK_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W) || !aligned16(out)) return PK_ERR_INVALID_ARG;
    const uint64_t limit = g_wait_limit_ns.load(std::memory_order_relaxed);
    if (use_pair())
        return pk::launch_dispatch_gemm_pair(false, x, nullptr, perm, expert_offsets, W, nullptr, T,
                                             k, D, E, D_expert, out, status_word,
                                             static_cast<cudaStream_t>(stream), limit);
    return pk::launch_dispatch_gemm_single(x, perm, expert_offsets, W, T, k, D, E, D_expert, out,
                                           status_word, static_cast<cudaStream_t>(stream), limit);
}

int pk_moe_dispatch_gemm_fp8(const uint8_t* xq, const float* sx, const int32_t* perm,
                             const int32_t* expert_offsets, const uint8_t* wq, const float* sw,
                             int32_t T, int32_t k, int32_t D, int32_t E, int32_t D_expert,
                             uint16_t* out, int32_t* status_word, void* stream) {
    if (T < 0 || k < 1 || E < 1 || D < 1 || D_expert < 1) return PK_ERR_INVALID_ARG;
    if ((D % 16) != 0 || (D_expert % 8) != 0) return PK_ERR_INVALID_ARG;
    const int64_t R = static_cast<int64_t>(T) * k;
    if (R >= (int64_t{1} << 31)) return PK_ERR_UNSUPPORTED;
    if (R == 0) return PK_OK;
    if (!xq || !sx || !perm || !expert_offsets || !wq || !sw || !out) return PK_ERR_INVALID_ARG;
    if (!aligned16(xq) || !aligned16(wq) || !aligned16(sw) || !aligned16(out))
        return PK_ERR_INVALID_ARG;
    if (pk_moe_fp8_weight_bytes(E, D, D_expert) >= (size_t{1} << 38)) return PK_ERR_UNSUPPORTED;
    const uint64_t limit = g_wait_limit_ns.load(std::memory_order_relaxed);
    if (use_pair())
        return pk::launch_dispatch_gemm_pair(true, xq, sx, perm, expert_offsets, wq, sw, T, k, D, E,
                                             D_expert, out, status_word,
                                             static_cast<cudaStream_t>(stream), limit);
    return pk::launch_dispatch_gemm_fp8_single(xq, sx, perm, expert_offsets, wq, sw, T, k, D, E,
                                               D_expert, out, status_word,
                                               static_cast<cudaStream_t>(stream), limit);
}

int pk_moe_quant_rows(const uint16_t* x, int32_t T, int32_t D, uint8_t* xq, float* sx,
                      void* stream) {
    if (T < 0 || D < 1 || (D % 8) != 0) return PK_ERR_INVALID_ARG;
    if (T == 0) return PK_OK;
    if (!x || !xq || !sx) return PK_ERR_INVALID_ARG;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(xq) & 7u) != 0) return PK_ERR_INVALID_ARG;
    cudaError_t err = pk::launch_quant_rows(x, T, D, xq, sx, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

size_t pk_moe_fp8_weight_bytes(int32_t E, int32_t D, int32_t N) {
    if (E < 1 || D < 1 || N < 1) return 0;
    return static_cast<size_t>(E) * static_cast<size_t>((N + 63) / 64) *
           static_cast<size_t>((D + 127) / 128) * 8192u;
}

int pk_moe_quant_weights(const uint16_t* W, int32_t E, int32_t D, int32_t N, uint8_t* wq,
                         float* sw, void* stream) {
    if (E < 1 || D < 1 || N < 1) return PK_ERR_INVALID_ARG;
    if (E > 65535) return PK_ERR_UNSUPPORTED;  // experts are a grid dimension
    if (!W || !wq || !sw) return PK_ERR_INVALID_ARG;
    // the GEMMs read W and wq by TMA (16-byte aligned) and sw as fp32
    if (!aligned16(W) || !aligned16(wq) || (reinterpret_cast<uintptr_t>(sw) & 3u) != 0)
        return PK_ERR_INVALID_ARG;
    cudaError_t err =
        pk::launch_quant_cols(W, E, D, N, wq, sw, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

int pk_moe_quant_rows_mx(const uint16_t* x, int32_t T, int32_t D, uint8_t* xq, uint8_t* sx,
                         void* stream) {
    if (T < 0 || D < 1 || (D % 32) != 0) return PK_ERR_INVALID_ARG;
    if (T == 0) return PK_OK;
    if (!x || !xq || !sx) return PK_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq)) return PK_ERR_INVALID_ARG;
    cudaError_t err = pk::launch_quant_rows_mx(x, T, D, xq, sx, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

size_t pk_moe_mx_weight_scale_bytes(int32_t E, int32_t D, int32_t N) {
    if (E < 1 || D < 128 || (D % 128) != 0 || N < 1) return 0;
    return pk::mx_weight_scale_bytes(E, D, N);
}

int pk_moe_quant_weights_mx(const uint16_t* W, int32_t E, int32_t D, int32_t N, uint8_t* wq,
                            uint8_t* swb, void* stream) {
    if (E < 1 || D < 1 || N < 1 || (D % 128) != 0 || (N % 8) != 0) return PK_ERR_INVALID_ARG;
    if (E > 65535) return PK_ERR_UNSUPPORTED;  // experts are a grid dimension
    if (!W || !wq || !swb) return PK_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(wq) || !aligned16(swb)) return PK_ERR_INVALID_ARG;
    cudaError_t err =
        pk::launch_quant_cols_mx(W, E, D, N, wq, swb, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

int pk_moe_dispatch_gemm_mxfp8(const uint8_t* xq, const uint8_t* sx, const int32_t* perm,
                               const int32_t* expert_offsets, const uint8_t* wq,
                               const uint8_t* swb, int32_t T, int32_t k, int32_t D, int32_t E,
                               int32_t D_expert, uint16_t* out, int32_t* status_word,
                               void* stream) {
    if (T < 0 || k < 1 || E < 1 || D < 1 || D_expert < 1) return PK_ERR_INVALID_ARG;
    if ((D % 128) != 0 || (D_expert % 8) != 0) return PK_ERR_INVALID_ARG;
    const int64_t R = static_cast<int64_t>(T) * k;
    if (R >= (int64_t{1} << 31)) return PK_ERR_UNSUPPORTED;
    if (R == 0) return PK_OK;
    if (!xq || !sx || !perm || !expert_offsets || !wq || !swb || !out) return PK_ERR_INVALID_ARG;
    if (!aligned16(xq) || !aligned16(wq) || !aligned16(swb) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(sx) & 3u) != 0)
        return PK_ERR_INVALID_ARG;
    if (pk_moe_fp8_weight_bytes(E, D, D_expert) >= (size_t{1} << 38)) return PK_ERR_UNSUPPORTED;
    return pk::launch_dispatch_gemm_mx(xq, sx, perm, expert_offsets, wq, swb, T, k, D, E, D_expert,
                                       out, status_word, static_cast<cudaStream_t>(stream),
                                       g_wait_limit_ns.load(std::memory_order_relaxed));
}

int pk_moe_grouped_gemm(const uint16_t* A, const int32_t* expert_offsets, const uint16_t* W,
                        int32_t R, int32_t K, int32_t N, int32_t E, uint16_t* out,
                        int32_t* status_word, void* stream) {
    if (R < 0 || K < 1 || N < 1 || E < 1) return PK_ERR_INVALID_ARG;
    if ((K % 8) != 0 || (N % 8) != 0) return PK_ERR_INVALID_ARG;
    if (R == 0) return PK_OK;
    if (!A || !expert_offsets || !W || !out) return PK_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(W) || !aligned16(out)) return PK_ERR_INVALID_ARG;
    return pk::launch_grouped_gemm(A, expert_offsets, W, R, K, N, E, out, status_word,
                                   static_cast<cudaStream_t>(stream),
                                   g_wait_limit_ns.load(std::memory_order_relaxed));
}

int pk_moe_grouped_gemm_fp8(const uint8_t* Aq, const float* sa, const int32_t* expert_offsets,
                            const uint8_t* wq, const float* sw, int32_t R, int32_t K, int32_t N,
                            int32_t E, uint16_t* out, int32_t* status_word, void* stream) {
    if (R < 0 || K < 1 || N < 1 || E < 1) return PK_ERR_INVALID_ARG;
    if ((K % 16) != 0 || (N % 8) != 0) return PK_ERR_INVALID_ARG;
    if (R == 0) return PK_OK;
    if (!Aq || !sa || !expert_offsets || !wq || !sw || !out) return PK_ERR_INVALID_ARG;
    if (!aligned16(Aq) || !aligned16(wq) || !aligned16(sw) || !aligned16(out))
        return PK_ERR_INVALID_ARG;
    if (pk_moe_fp8_weight_bytes(E, K, N) >= (size_t{1} << 38)) return PK_ERR_UNSUPPORTED;
    return pk::launch_grouped_gemm_fp8(Aq, sa, expert_offsets, wq, sw, R, K, N, E, out,
                                       status_word, static_cast<cudaStream_t>(stream),
                                       g_wait_limit_ns.load(std::memory_order_relaxed));
}

int pk_moe_router_topk(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_idx,
                       float* gates, void* stream) {
    if (T < 0 || E < 1 || k < 1 || k > E || k > 32) return PK_ERR_INVALID_ARG;
    if (E > PK_ROUTER_MAX_EXPERTS) return PK_ERR_UNSUPPORTED;
    if (T > 0 && (!logits || !topk_idx)) return PK_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * E >= (int64_t{1} << 40)) return PK_ERR_UNSUPPORTED;
    cudaError_t err = pk::launch_router_topk(logits, T, E, k, topk_idx, gates,
                                             static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

int pk_moe_combine(const uint16_t* src, const int32_t* inv_perm, const float* gates, int32_t T,
                   int32_t k, int32_t C, uint16_t* y, int32_t* status_word, void* stream) {
    if (T < 0 || k < 1 || C < 1 || (C % 8) != 0) return PK_ERR_INVALID_ARG;
    const int64_t R = static_cast<int64_t>(T) * k;
    if (R >= (int64_t{1} << 31)) return PK_ERR_UNSUPPORTED;
    if (T == 0) return PK_OK;
    if (!src || !inv_perm || !y) return PK_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(y)) return PK_ERR_INVALID_ARG;
    cudaError_t err = pk::launch_combine(src, inv_perm, gates, T, k, C, y, status_word,
                                         static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

int pk_moe_route_kernel_launches(int32_t T, int32_t k, int32_t E) {
    if (T < 0 || k < 1 || E < 1) return -1;
    return pk::route_kernel_launches(static_cast<int64_t>(T) * k, E);
}

int pk_moe_set_gemm_kernel(int kernel) {
    if (kernel != PK_GEMM_KERNEL_AUTO && kernel != PK_GEMM_KERNEL_SINGLE &&
        kernel != PK_GEMM_KERNEL_PAIR)
        return PK_ERR_INVALID_ARG;
    g_gemm_kernel.store(kernel, std::memory_order_relaxed);
    return PK_OK;
}

void pk_moe_set_wait_limit_ns(uint64_t limit_ns) {
    g_wait_limit_ns.store(limit_ns ? limit_ns : kDefaultWaitLimitNs, std::memory_order_relaxed);
}

void pk_debug_stall_gemm(int32_t cta, int64_t kstep) { pk::set_debug_stall(cta, kstep); }

int pk_debug_bounded_wait(int32_t* status_word, uint64_t limit_ns, void* stream) {
    if (!status_word || limit_ns == 0) return PK_ERR_INVALID_ARG;
    cudaError_t err =
        pk::launch_bounded_wait_probe(status_word, limit_ns, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

}  // extern "C"
