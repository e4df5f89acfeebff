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
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "pk_internal.h"

namespace {

// 1 MiB of int32 counters: ceil(T*k / 2048) * E must not exceed this.
constexpr size_t kNoAllocScratchInts = PK_NOALLOC_SCRATCH_BYTES / sizeof(int32_t);

__device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchInts];

// Device address of g_route_scratch in the current CUDA context. In host code
// the symbol's name is only a host-side stand-in, never a device address. The
// address belongs to the context that loaded the library's module, so it is
// cached per device together with that context's unique id (a context made
// anew, e.g. after cudaDeviceReset, has a new id and its own address), and
// it is never looked up during stream capture, where loading a module is not
// allowed.
struct ScratchSlot {
    unsigned long long ctx_id = 0;
    int32_t* addr = nullptr;
};
ScratchSlot g_scratch[64];
std::mutex g_scratch_mu;

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_fn_once;

// Unique id of the current context; false if there is none or the driver
// entry points are unavailable.
bool current_ctx_id(unsigned long long* id) {
    std::call_once(g_ctx_fn_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    CUcontext ctx = nullptr;
    if (!g_ctx_current || !g_ctx_id || g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return false;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

int scratch_for_current_context(cudaStream_t stream, int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PK_ERR_CUDA;
    unsigned long long id = 0;
    const bool have_id = current_ctx_id(&id);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchSlot& slot = g_scratch[dev];
    if (have_id && slot.addr && slot.ctx_id == id) {
        *out = slot.addr;
        return PK_OK;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return PK_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return PK_ERR_CAPTURE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
        return PK_ERR_CUDA;
    // the lookup made the context current if there was none yet
    if (!have_id && !current_ctx_id(&id)) return PK_ERR_CUDA;
    slot.ctx_id = id;
    slot.addr = static_cast<int32_t*>(p);
    *out = slot.addr;
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

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* scratch = nullptr;
    const int rc = scratch_for_current_context(s, &scratch);
    if (rc != PK_OK) return rc;
    if (pk::launch_route_counts(topk_idx, static_cast<int32_t>(R), E, expert_counts,
                                expert_offsets, scratch, status_word, s) != cudaSuccess)
        return PK_ERR_CUDA;
    if (pk::launch_build_perm(topk_idx, static_cast<int32_t>(R), E, scratch, perm, inv_perm,
                              status_word, s) != cudaSuccess)
        return PK_ERR_CUDA;
    return PK_OK;
}
