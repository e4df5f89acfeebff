// Routing for callers that cannot allocate device memory.
//
// pk_moe_route_counts and pk_moe_build_perm take a workspace from the caller.
// Some callers cannot provide one: a host program that hands all device
// memory to its own pool at start-up, a plug-in inside an inference runtime
// whose allocator it may not bypass, or code on a latency-critical path where
// cudaMalloc's implicit device synchronisation is not acceptable. For them,
// pk_moe_route_noalloc runs the same three routing kernels with their
// per-chunk counters in a fixed array that lives in this library's device
// image (every GPU that loads the library keeps it until the process exits).
//
// The array is shared by every call in the process: it keeps the last call's
// contents, and each call rewrites every counter it later reads (the histogram
// kernel writes all E counters of every chunk before anything reads them), so
// nothing needs clearing between calls. Calls that overlap on the GPU (on
// different streams, or from different host threads) use the same array and
// race; order them on one stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pk_internal.h"

namespace {

// 1 MiB of int32 counters: ceil(T*k / 2048) * E must not exceed this.
constexpr size_t kNoAllocScratchInts = PK_NOALLOC_SCRATCH_BYTES / sizeof(int32_t);

__device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchInts];

// Device address of g_route_scratch, looked up once per device. In host code
// the symbol's name is only a host-side stand-in, never a device address.
int32_t* g_scratch_addr[64] = {nullptr};
std::mutex g_scratch_mu;

int scratch_for_current_device(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PK_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
            return PK_ERR_CUDA;
        g_scratch_addr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_addr[dev];
    return PK_OK;
}

}  // namespace

extern "C" int pk_moe_route_noalloc(const int32_t* topk_idx, int32_t T, int32_t k, int32_t E,
                                    int32_t* expert_counts, int32_t* expert_offsets,
                                    int32_t* perm, int32_t* inv_perm, int32_t* status_word,
                                    void* stream) {
    if (T < 0 || k < 1 || E < 1 || k > E || !expert_offsets) return PK_ERR_INVALID_ARG;
    if (E > PK_MAX_EXPERTS) return PK_ERR_UNSUPPORTED;
    const int64_t R = static_cast<int64_t>(T) * k;
    if (R >= (int64_t{1} << 31)) return PK_ERR_UNSUPPORTED;
    if (R > 0 && (!topk_idx || !perm)) return PK_ERR_INVALID_ARG;
    const int64_t need = static_cast<int64_t>(pk::route_blocks(R)) * E;
    if (need > static_cast<int64_t>(kNoAllocScratchInts)) return PK_ERR_UNSUPPORTED;

    int32_t* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != PK_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pk::launch_route_counts(topk_idx, static_cast<int32_t>(R), E, expert_counts,
                                expert_offsets, scratch, status_word, s) != cudaSuccess)
        return PK_ERR_CUDA;
    if (pk::launch_build_perm(topk_idx, static_cast<int32_t>(R), E, scratch, perm, inv_perm,
                              status_word, s) != cudaSuccess)
        return PK_ERR_CUDA;
    return PK_OK;
}
