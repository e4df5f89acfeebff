// Routing kernels: expert histogram, exclusive scan and the stable
// (expert, token, slot) permutation of the routed rows -- the "dispatch" half
// of the token-dispatch + GEMM of "Loads and Loads of Fluffy Kittens"
// ("Key claims", Fig. 17), restated for one device.
//
// The flat routing array topk_idx[T*k] is cut into chunks of kRouteChunk
// entries, one block per chunk, in flat order. Workspace holds one row of E
// counters per chunk:
//   k_route_hist   row b = histogram of chunk b;
//   k_route_scan   counts, offsets = exclusive scan of the column sums, and
//                  row b rewritten in place to the first output position of
//                  chunk b's entries of each expert:
//                    base[b][e] = offsets[e] + sum_{b' < b} hist[b'][e];
//   k_route_small  both of the above in one block of 1024 threads, for
//                  routing arrays of at most two chunks (one launch instead
//                  of two; on larger arrays one SM's __match_any_sync rate
//                  makes it slower than the spread-out histogram);
//   k_build_perm   each warp of block b owns a contiguous run of the chunk
//                  (2 entries per lane in 32-warp blocks when 32 warp
//                  histograms of E counters fit 48 KiB, else 8 per lane in
//                  8-warp blocks; loaded once into registers); a
//                  per-warp histogram and a scan over warps give every warp
//                  its first position per expert, then warps walk their runs
//                  32 entries at a time and rank equal experts inside a warp
//                  with __match_any_sync. Positions follow flat order, so the
//                  result is unique and needs no atomics.
//
// All four are launched with programmatic stream serialisation and call
// grid_dep_wait() before their first global access: a kernel's launch and
// shared-memory set-up overlap the tail of the kernel ahead of it, and
// nothing else does. The histogram kernels load all their entries before
// counting any (one memory round trip per block); the scan copies the chunk
// rows into shared memory in one coalesced pass when they fit.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pk_internal.h"
#include "pk_ptx.cuh"

namespace pk {

// Entries of one chunk held by each thread of the histogram kernel.
constexpr int kHistPer = kRouteChunk / kRouteThreads;
static_assert(kRouteChunk % kRouteThreads == 0, "a chunk is a whole number of block rounds");

__global__ void __launch_bounds__(kRouteThreads)
    k_route_hist(const int32_t* __restrict__ topk, int32_t R, int32_t E,
                 int32_t* __restrict__ blockcnt, int32_t* status) {
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += kRouteThreads) hist[e] = 0;
    // topk may come from the kernel ahead in the stream, and the chunk rows
    // may still be read by the previous routing call: touch neither before.
    grid_dep_wait();
    grid_dep_release();
    const int64_t beg = static_cast<int64_t>(blockIdx.x) * kRouteChunk;
    const uint32_t lane = threadIdx.x & 31;
    // All of this thread's entries are loaded before any is counted, so the
    // block waits for one round trip to memory instead of kHistPer.
    int32_t ent[kHistPer];
    bool bad = false;
#pragma unroll
    for (int it = 0; it < kHistPer; ++it) {
        const int64_t i = beg + it * kRouteThreads + threadIdx.x;
        int32_t e = -1;
        if (i < R) {
            e = __ldg(topk + i);
            if (e < 0 || e >= E) {
                bad = true;
                e = -1;
            }
        }
        ent[it] = e;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < kHistPer; ++it) {
        const int32_t e = ent[it];
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == static_cast<uint32_t>(__ffs(peers) - 1))
            atomicAdd(&hist[e], __popc(peers));
    }
    if (bad) report(status, PK_ERR_BAD_INDEX);
    __syncthreads();
    int32_t* row = blockcnt + static_cast<int64_t>(blockIdx.x) * E;
    for (int e = threadIdx.x; e < E; e += kRouteThreads) row[e] = hist[e];
}

constexpr int kScanThreads = 1024;

// Exclusive scan of v[0, n) into out[0, n) by one block of kScanThreads
// threads (each thread a run of consecutive values, a warp shuffle scan and a
// scan of the 32 warp sums); returns the total to every thread. wsum: [32].
__device__ int32_t block_exclusive_scan(const int32_t* v, int32_t* out, int n, int32_t* wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + kScanThreads - 1) / kScanThreads;
    const int b0 = min(tid * per, n), b1 = min(b0 + per, n);
    int32_t local = 0;
    for (int i = b0; i < b1; ++i) local += v[i];
    int32_t incl = local;
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t w = wsum[lane];
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += t;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    int32_t run = (warp > 0 ? wsum[warp - 1] : 0) + incl - local;
    for (int i = b0; i < b1; ++i) {
        out[i] = run;
        run += v[i];
    }
    const int32_t total = wsum[31];
    __syncthreads();
    return total;
}

// Shared memory the scan may take to hold every chunk row while it reads them
// twice (column sums, then starting positions); larger arrays of chunk rows
// are read from global memory in place.
constexpr size_t kScanStageSmem = 96 * 1024;

inline size_t scan_smem_bytes(int32_t nblk, int32_t E, bool staged) {
    const size_t base = sizeof(int32_t) * (2 * static_cast<size_t>(E) + 32);
    return staged ? base + sizeof(int32_t) * static_cast<size_t>(nblk) * E : base;
}

inline bool scan_staged(int32_t nblk, int32_t E) {
    return scan_smem_bytes(nblk, E, true) <= kScanStageSmem;
}

// Shared memory: tot [E], offs [E], wsum [32], then (staged) rows [nblk][E].
__global__ void __launch_bounds__(kScanThreads)
    k_route_scan(int32_t* __restrict__ blockcnt, int32_t nblk, int32_t E, int32_t* counts,
                 int32_t* __restrict__ offsets, int32_t staged) {
    extern __shared__ int32_t sm[];
    int32_t* tot = sm;            // [E]
    int32_t* offs = sm + E;       // [E]
    int32_t* wsum = sm + 2 * E;   // [32]
    int32_t* rows = sm + 2 * E + 32;
    const int tid = threadIdx.x;
    grid_dep_wait();
    grid_dep_release();

    // One coalesced pass brings every chunk row into shared memory: the
    // loads are independent, so they overlap instead of walking the chunks
    // one dependent load at a time per expert.
    const int64_t n = static_cast<int64_t>(nblk) * E;
    if (staged) {
        for (int64_t i = tid; i < n; i += kScanThreads) rows[i] = blockcnt[i];
        __syncthreads();
    }
    const int32_t* src = staged ? rows : blockcnt;

    for (int e = tid; e < E; e += kScanThreads) {
        int32_t s = 0;
        for (int b = 0; b < nblk; ++b) s += src[static_cast<int64_t>(b) * E + e];
        tot[e] = s;
        if (counts) counts[e] = s;
    }
    __syncthreads();
    const int32_t total = block_exclusive_scan(tot, offs, E, wsum);
    for (int e = tid; e < E; e += kScanThreads) offsets[e] = offs[e];
    if (tid == 0) offsets[E] = total;

    // Per-chunk starting positions, written over the chunk histograms.
    for (int e = tid; e < E; e += kScanThreads) {
        int32_t r = offs[e];
        for (int b = 0; b < nblk; ++b) {
            const int64_t i = static_cast<int64_t>(b) * E + e;
            const int32_t cnt = src[i];
            blockcnt[i] = r;
            r += cnt;
        }
    }
}

// k_route_small takes routing arrays of at most this many chunks whose
// histograms (nblk * E ints) fit this much shared memory.
constexpr int kRouteSmallChunks = 2;
constexpr size_t kRouteSmallSmem = 96 * 1024;
// Entries per thread of k_route_small.
constexpr int kSmallPer = kRouteSmallChunks * kRouteChunk / kScanThreads;
static_assert(kRouteSmallChunks * kRouteChunk % kScanThreads == 0, "whole rounds");

// Chunk histograms, counts, offsets and chunk starting positions in one block.
// Shared memory: hist [nblk][E], tot [E], offs [E], wsum [32].
__global__ void __launch_bounds__(kScanThreads)
    k_route_small(const int32_t* __restrict__ topk, int32_t R, int32_t E, int32_t nblk,
                  int32_t* __restrict__ blockbase, int32_t* counts, int32_t* __restrict__ offsets,
                  int32_t* status) {
    extern __shared__ int32_t sm[];
    int32_t* hist = sm;
    int32_t* tot = hist + static_cast<int64_t>(nblk) * E;
    int32_t* offs = tot + E;
    int32_t* wsum = offs + E;
    const uint32_t lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < nblk * E; i += blockDim.x) hist[i] = 0;
    grid_dep_wait();
    grid_dep_release();
    // every entry loaded before any is counted (one round trip to memory)
    int32_t ent[kSmallPer];
    bool bad = false;
#pragma unroll
    for (int it = 0; it < kSmallPer; ++it) {
        const int i = it * kScanThreads + threadIdx.x;
        int32_t e = -1;
        if (i < R) {
            e = __ldg(topk + i);
            if (e < 0 || e >= E) {
                bad = true;
                e = -1;
            }
        }
        ent[it] = e;
    }
    __syncthreads();
    // 32 consecutive entries always lie in one chunk (kRouteChunk % 32 == 0)
#pragma unroll
    for (int it = 0; it < kSmallPer; ++it) {
        const int i = it * kScanThreads + threadIdx.x;
        const int32_t e = ent[it];
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == static_cast<uint32_t>(__ffs(peers) - 1))
            atomicAdd(&hist[(i / kRouteChunk) * E + e], __popc(peers));
    }
    if (bad) report(status, PK_ERR_BAD_INDEX);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t s = 0;
        for (int b = 0; b < nblk; ++b) s += hist[b * E + e];
        tot[e] = s;
        if (counts) counts[e] = s;
    }
    __syncthreads();
    const int32_t total = block_exclusive_scan(tot, offs, E, wsum);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        offsets[e] = offs[e];
        int32_t r = offs[e];
        for (int b = 0; b < nblk; ++b) {
            blockbase[static_cast<int64_t>(b) * E + e] = r;
            r += hist[b * E + e];
        }
    }
    if (threadIdx.x == 0) offsets[E] = total;
}

template <int kWarps>
__global__ void __launch_bounds__(kWarps * 32)
    k_build_perm(const int32_t* __restrict__ topk, int32_t R, int32_t E,
                 const int32_t* __restrict__ blockbase, int32_t* __restrict__ perm,
                 int32_t* __restrict__ inv_perm, int32_t* status) {
    extern __shared__ int32_t wpos[];  // [kWarps][E]
    static_assert(kRouteChunk % (kWarps * 32) == 0, "whole 32-entry rounds per warp");
    constexpr int kPerWarp = kRouteChunk / kWarps;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) wpos[i] = 0;
    grid_dep_wait();
    grid_dep_release();
    // This block's starting position of expert threadIdx.x, fetched now so
    // that its latency overlaps the loads and the warp histograms below.
    const int32_t* bb = blockbase + static_cast<int64_t>(blockIdx.x) * E;
    const int32_t bb_first = static_cast<int>(threadIdx.x) < E ? bb[threadIdx.x] : 0;
    __syncthreads();

    const int64_t wbeg = static_cast<int64_t>(blockIdx.x) * kRouteChunk +
                         static_cast<int64_t>(warp) * kPerWarp;
    const int64_t wend = min(wbeg + kPerWarp, static_cast<int64_t>(R));
    int32_t* my = wpos + warp * E;

    // This lane's entries of the warp's run, loaded once (-1: none or invalid).
    constexpr int kIter = kPerWarp / 32;
    int32_t ent[kIter];
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const int64_t i = wbeg + it * 32 + lane;
        int32_t e = -1;
        if (i < wend) {
            e = __ldg(topk + i);
            if (e < 0 || e >= E) e = -1;
        }
        ent[it] = e;
    }

    // Pass 1: histogram of this warp's run.
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const int32_t e = ent[it];
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // Pass 2: first position of every warp's entries, per expert.
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t r = e == static_cast<int>(threadIdx.x) ? bb_first : bb[e];
        for (int w = 0; w < kWarps; ++w) {
            const int32_t c = wpos[w * E + e];
            wpos[w * E + e] = r;
            r += c;
        }
    }
    __syncthreads();

    // Pass 3: scatter in flat order.
    bool bad = false;
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const int64_t i = wbeg + it * 32 + lane;
        const int32_t e = ent[it];
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0) {
            const int32_t pos = my[e] + __popc(peers & lt_mask);
            if (pos >= 0 && pos < R) {
                perm[pos] = static_cast<int32_t>(i);
                if (inv_perm) inv_perm[i] = pos;
            } else {
                bad = true;
            }
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
    }
    if (bad) report(status, PK_ERR_BAD_INDEX);
}

// Warps of the permutation kernel's wide form (1024 threads).
constexpr int kPermWideWarps = 32;

namespace {
int g_perm_smem_set[64] = {0};
int g_small_smem_set[64] = {0};
int g_scan_smem_set[64] = {0};

// Raises a kernel's dynamic shared-memory limit to `bytes`, once per device.
template <typename Kernel>
cudaError_t allow_smem(Kernel kern, int* done, size_t bytes) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(bytes));
    if (err == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
    return err;
}

// Launches a routing kernel with programmatic stream serialisation: its
// blocks may be scheduled while the kernel ahead of it is finishing. Every
// routing kernel calls grid_dep_wait() before its first access to global
// memory, so results are the same as with a plain launch; what overlaps is
// the launch itself and the kernel's shared-memory set-up.
template <typename... Params, typename... Args>
cudaError_t launch_chained(void (*kern)(Params...), int grid, int block, size_t smem,
                           cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}
}  // namespace

cudaError_t launch_route_counts(const int32_t* topk, int32_t R, int32_t E, int32_t* counts,
                                int32_t* offsets, int32_t* blockbase, int32_t* status,
                                cudaStream_t stream) {
    const int nblk = route_blocks(R);
    const size_t small_smem = sizeof(int32_t) * (static_cast<size_t>(nblk) * E + 2 * E + 32);
    cudaError_t err;
    if (nblk > 0 && nblk <= kRouteSmallChunks && small_smem <= kRouteSmallSmem) {
        if (small_smem > 48 * 1024) {
            err = allow_smem(k_route_small, g_small_smem_set, kRouteSmallSmem);
            if (err != cudaSuccess) return err;
        }
        return launch_chained(k_route_small, 1, kScanThreads, small_smem, stream, topk, R, E, nblk,
                              blockbase, counts, offsets, status);
    }
    if (nblk > 0) {
        err = launch_chained(k_route_hist, nblk, kRouteThreads, sizeof(int32_t) * E, stream, topk,
                             R, E, blockbase, status);
        if (err != cudaSuccess) return err;
    }
    const bool staged = scan_staged(nblk, E);
    const size_t scan_smem = scan_smem_bytes(nblk, E, staged);
    if (scan_smem > 48 * 1024) {
        err = allow_smem(k_route_scan, g_scan_smem_set, kScanStageSmem);
        if (err != cudaSuccess) return err;
    }
    return launch_chained(k_route_scan, 1, kScanThreads, scan_smem, stream, blockbase, nblk, E,
                          counts, offsets, static_cast<int32_t>(staged));
}

int route_kernel_launches(int64_t R, int32_t E) {
    if (R <= 0) return 1;  // the scan alone writes the zero offsets
    const int nblk = route_blocks(R);
    const size_t small_smem = sizeof(int32_t) * (static_cast<size_t>(nblk) * E + 2 * E + 32);
    return nblk <= kRouteSmallChunks && small_smem <= kRouteSmallSmem ? 2 : 3;
}

cudaError_t launch_build_perm(const int32_t* topk, int32_t R, int32_t E,
                              const int32_t* blockbase, int32_t* perm, int32_t* inv_perm,
                              int32_t* status, cudaStream_t stream) {
    const int nblk = route_blocks(R);
    if (nblk == 0) return cudaSuccess;
    // 32 warps (2 entries per lane: four rounds of __match_any_sync ranking
    // instead of sixteen) when their histograms fit the default 48 KiB.
    const size_t smem32 = sizeof(int32_t) * kPermWideWarps * static_cast<size_t>(E);
    if (smem32 <= 48 * 1024)
        return launch_chained(k_build_perm<kPermWideWarps>, nblk, kPermWideWarps * 32, smem32,
                              stream, topk, R, E, blockbase, perm, inv_perm, status);
    const size_t smem = sizeof(int32_t) * kRouteWarps * static_cast<size_t>(E);
    if (smem > 48 * 1024) {
        const cudaError_t err = allow_smem(k_build_perm<kRouteWarps>, g_perm_smem_set,
                                           sizeof(int32_t) * kRouteWarps * PK_MAX_EXPERTS);
        if (err != cudaSuccess) return err;
    }
    return launch_chained(k_build_perm<kRouteWarps>, nblk, kRouteThreads, smem, stream, topk, R, E,
                          blockbase, perm, inv_perm, status);
}

}  // namespace pk
