// Token dispatch fused with the per-expert up-projection GEMM on sm_103a:
//   out[j, :] = x[perm[j] / k, :] @ W[e(j)]   for j in expert e's segment
// -- the "token-dispatch + GEMM" of "Loads and Loads of Fluffy Kittens"
// ("Key claims", Fig. 17) on one device. What carries over from the pages is
// their intra-SM overlap (section "Using the Right Overlapping Schedule"):
// a producer warp moves tiles with TMA while the tensor cores stay busy.
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0     producer: per K-step of 64, TMA-loads the W_e tile [64 x BN]
//              (four 64x64 boxes, 128-byte swizzle) and gathers the unit's
//              routed x rows straight into 128-byte-swizzled shared memory
//              with four-row TMA gathers (lane l fetches rows 4l..4l+3).
//   warp 1     MMA issuer (one thread): tcgen05.mma M=128 x N=BN x K=16 per
//              m-tile into fp32 accumulators in TMEM; commits free the stage.
//   warps 2-5  epilogue: tcgen05.ld from TMEM, bf16 round-to-nearest-even,
//              masked 16-byte stores of the valid rows and columns.
// A 3-stage shared-memory ring (full/empty mbarriers) connects producer and
// MMA; an accumulator barrier pair connects MMA and epilogue.
//
// Work unit = (expert e, n-tile of BN <= 256 columns, group of up to two
// 128-row m-tiles). Both m-tiles of a unit share every W tile it loads, so an
// expert with at most 256 rows streams its W_e exactly once. Units are
// numbered expert-major (e, n, group) and dealt round-robin to the CTAs, so
// units that share a W tile or the same gathered rows run at the same time
// and meet in L2. Experts with no rows contribute no units.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "pk_internal.h"
#include "pk_ptx.cuh"

namespace pk {
namespace dg {

constexpr int BM = 128;                      // rows per m-tile (MMA M)
constexpr int BK = 64;                       // K per stage: one 128-byte swizzle row of bf16
constexpr int BN = 256;                      // widest n-tile (MMA N)
constexpr int MT = 2;                        // m-tiles (accumulators) per unit
constexpr int STAGES = 3;
constexpr int B_BOX = 64;                    // W box: 64 columns x 64 rows
constexpr int B_BOX_BYTES = B_BOX * BK * 2;  // 8 KiB
constexpr int B_BYTES = BK * BN * 2;         // 32 KiB
constexpr int A_BYTES = BM * BK * 2;         // 16 KiB
constexpr int STAGE_BYTES = B_BYTES + MT * A_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;          // MT accumulators of BN fp32 columns
constexpr int UMMA_K = 16;

struct Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + static_cast<int>(sizeof(Ctrl)) + 64;

struct Unit {
    int e;        // expert
    int row0;     // first sorted row of the unit
    int rows;     // valid rows (<= MT * BM)
    int mtiles;   // ceil(rows / BM)
    int n0;       // first output column
    int bn;       // n-tile width: a multiple of 64, <= BN
};

// Walks the expert-major unit numbering; u must not decrease between calls.
struct Walker {
    const int32_t* off;
    int E, R, De, ntiles;
    int e;
    int64_t base;  // units of experts < e
    int lo, rows, groups;
    int64_t units;

    __device__ void init(const int32_t* o, int E_, int R_, int De_) {
        off = o; E = E_; R = R_; De = De_;
        ntiles = (De + BN - 1) / BN;
        e = 0; base = 0;
        load();
    }
    __device__ void load() {
        if (e >= E) { units = 0; return; }
        int a = __ldg(off + e), b = __ldg(off + e + 1);
        a = min(max(a, 0), R);
        b = min(max(b, a), R);
        lo = a;
        rows = b - a;
        const int mt = (rows + BM - 1) / BM;
        groups = (mt + MT - 1) / MT;
        units = static_cast<int64_t>(groups) * ntiles;
    }
    __device__ bool find(int64_t u, Unit& U) {
        while (e < E && u >= base + units) {
            base += units;
            ++e;
            load();
        }
        if (e >= E) return false;
        const int l = static_cast<int>(u - base);
        const int n = l / groups, g = l - n * groups;
        U.e = e;
        U.row0 = lo + g * (MT * BM);
        U.rows = min(MT * BM, rows - g * (MT * BM));
        U.mtiles = (U.rows + BM - 1) / BM;
        U.n0 = n * BN;
        U.bn = min(BN, (De - U.n0 + B_BOX - 1) / B_BOX * B_BOX);
        return true;
    }
};

// One lane waits; the warp learns the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                          uint64_t limit) {
    bool ok = true;
    if (lane_id() == 0) ok = mbar_wait(bar, parity, abort, limit);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}

__device__ __forceinline__ void fail(volatile int* abort, int32_t* status) {
    report(status, PK_ERR_TIMEOUT);
    *abort = 1;
}

__global__ void __launch_bounds__(THREADS, 1)
    k_dispatch_gemm(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                    const int32_t* __restrict__ perm, const int32_t* __restrict__ offsets,
                    uint16_t* __restrict__ out, int32_t T, int32_t k, int32_t D, int32_t E,
                    int32_t De, int32_t* status, uint64_t limit) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (sbase - raw);
    Ctrl* ctl = reinterpret_cast<Ctrl*>(base_ptr + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int R = T * k;
    const int nk = (D + BK - 1) / BK;

    const uint32_t full0 = smem_addr(&ctl->full[0]);
    const uint32_t empty0 = smem_addr(&ctl->empty[0]);
    const uint32_t acc_full = smem_addr(&ctl->acc_full);
    const uint32_t acc_empty = smem_addr(&ctl->acc_empty);
    const uint32_t drain = smem_addr(&ctl->drain);
    volatile int* abort = &ctl->abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(drain, 1);
        ctl->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&xmap);
        prefetch_tensormap(&wmap);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        const uint64_t pol_w = policy_evict_first();  // each W tile is needed once
        const uint64_t pol_x = policy_evict_last();   // rows are re-read by other n-tiles
        Walker wk;
        wk.init(offsets, E, R, De);
        int stage = 0;
        uint32_t phase = 0, issued = 0, issued_par = 0;
        bool ok = true, bad = false;
        for (int64_t u = blockIdx.x; ok; u += gridDim.x) {
            Unit U;
            if (!wk.find(u, U)) break;
            int rr[MT][4];
            bool go[MT];
            uint32_t bytes = static_cast<uint32_t>(U.bn / B_BOX) * B_BOX_BYTES;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int p0 = mt * BM + 4 * lane;
                go[mt] = mt < U.mtiles && p0 < U.rows;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    int t = 0;
                    if (go[mt]) {
                        const int p = (p0 + i < U.rows) ? p0 + i : p0;
                        int f = __ldg(perm + U.row0 + p);
                        if (f < 0 || f >= R) {
                            bad = true;
                            f = 0;
                        }
                        t = f / k;
                    }
                    rr[mt][i] = t;
                }
                const int vm = min(max(U.rows - mt * BM, 0), BM);
                bytes += static_cast<uint32_t>((vm + 3) / 4) * (4 * BK * 2);
            }
            for (int ks = 0; ks < nk; ++ks) {
                if (!warp_wait(empty0 + 8 * stage, phase ^ 1u, abort, limit)) {
                    if (lane == 0) fail(abort, status);
                    ok = false;
                    break;
                }
                const uint32_t full = full0 + 8 * stage;
                if (lane == 0) mbar_arrive_expect_tx(full, bytes);
                __syncwarp();
                const uint32_t sb = sbase + stage * STAGE_BYTES;
                if (lane < U.bn / B_BOX)
                    tma_load_3d(sb + lane * B_BOX_BYTES, &wmap, U.n0 + lane * B_BOX, ks * BK, U.e,
                                full, pol_w);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
                    if (go[mt])
                        tma_gather4(sb + B_BYTES + mt * A_BYTES + lane * (4 * BK * 2), &xmap,
                                    ks * BK, rr[mt][0], rr[mt][1], rr[mt][2], rr[mt][3], full,
                                    pol_x);
                issued |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (bad) report(status, PK_ERR_BAD_INDEX);
        // Every copy this warp started must land before the CTA may exit.
        if (lane == 0)
            for (int s = 0; s < STAGES; ++s)
                if ((issued >> s) & 1u) mbar_wait(full0 + 8 * s, (issued_par >> s) & 1u, nullptr, limit);
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA
        if (lane == 0) {
            Walker wk;
            wk.init(offsets, E, R, De);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok; u += gridDim.x) {
                Unit U;
                if (!wk.find(u, U)) break;
                if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort, limit)) {
                    fail(abort, status);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t idesc = idesc_bf16_f32(BM, U.bn, true);
                for (int ks = 0; ks < nk; ++ks) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort, limit)) {
                        fail(abort, status);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sb = sbase + stage * STAGE_BYTES;
                    for (int mt = 0; mt < U.mtiles; ++mt) {
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            // A: K-major, rows 128 B apart, 8-row groups 1024 B apart;
                            // a K step of 16 moves 32 B inside the swizzled row.
                            const uint64_t a = sdesc_sw128(
                                sb + B_BYTES + mt * A_BYTES + kk * (UMMA_K * 2), 16, 1024);
                            // B: MN-major (W rows are N-contiguous), 64-column blocks
                            // 8 KiB apart (LBO), 8-row K groups 1024 B apart (SBO);
                            // a K step of 16 moves 16 rows = 2 KiB.
                            const uint64_t b = sdesc_sw128(sb + kk * (UMMA_K * 128), B_BOX_BYTES, 1024);
                            mma_bf16(tmem + static_cast<uint32_t>(mt * BN), a, b, idesc,
                                     (ks | kk) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(empty0 + 8 * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(acc_full);
                acc_phase ^= 1u;
            }
            // All MMAs this thread issued must finish before TMEM is freed.
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, limit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        Walker wk;
        wk.init(offsets, E, R, De);
        uint32_t acc_phase = 0;
        for (int64_t u = blockIdx.x;; u += gridDim.x) {
            Unit U;
            if (!wk.find(u, U)) break;
            if (!warp_wait(acc_full, acc_phase, abort, limit)) {
                if (lane == 0) fail(abort, status);
                break;
            }
            tc_fence_after_sync();
            for (int mt = 0; mt < U.mtiles; ++mt) {
                const int rbase = mt * BM + q * 32;
                if (rbase >= U.rows) continue;  // warp-uniform
                const int r = rbase + lane;
                const bool valid = r < U.rows;
                uint16_t* orow = out + static_cast<int64_t>(U.row0 + r) * De;
                const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(mt * BN);
                for (int c = 0; c < U.bn / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_wait_ld();
                    const int col0 = U.n0 + c * 32;
                    if (valid) {
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            if (col0 + g * 8 < De) {
                                uint4 pkd;
                                uint32_t* w = reinterpret_cast<uint32_t*>(&pkd);
#pragma unroll
                                for (int h = 0; h < 4; ++h) {
                                    __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                        __uint_as_float(v[g * 8 + 2 * h]),
                                        __uint_as_float(v[g * 8 + 2 * h + 1]));
                                    w[h] = *reinterpret_cast<uint32_t*>(&b2);
                                }
                                *reinterpret_cast<uint4*>(orow + col0 + g * 8) = pkd;
                            }
                        }
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            acc_phase ^= 1u;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace dg

// ------------------------------------------------------------------ host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

struct DevInfo {
    int sms = 0;
    bool attr_set = false;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

}  // namespace

int launch_dispatch_gemm(const uint16_t* x, const int32_t* perm, const int32_t* offsets,
                         const uint16_t* W, int32_t T, int32_t k, int32_t D, int32_t E,
                         int32_t De, uint16_t* out, int32_t* status, cudaStream_t stream,
                         uint64_t wait_limit_ns) {
    using namespace dg;
    auto enc = encoder();
    if (!enc) return PK_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PK_ERR_CUDA;
    int sms;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        DevInfo& di = g_dev[dev];
        if (!di.attr_set) {
            if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return PK_ERR_CUDA;
            if (cudaFuncSetAttribute(k_dispatch_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SMEM_BYTES) != cudaSuccess)
                return PK_ERR_CUDA;
            di.attr_set = true;
        }
        sms = di.sms;
    }

    CUtensorMap xmap, wmap;
    {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
        cuuint32_t box[2] = {BK, 1};
        cuuint32_t es[2] = {1, 1};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PK_ERR_UNSUPPORTED;
    }
    {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(De), static_cast<cuuint64_t>(D),
                              static_cast<cuuint64_t>(E)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(De) * 2,
                                 static_cast<cuuint64_t>(D) * static_cast<cuuint64_t>(De) * 2};
        cuuint32_t box[3] = {B_BOX, BK, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(W), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PK_ERR_UNSUPPORTED;
    }
    k_dispatch_gemm<<<sms, THREADS, SMEM_BYTES, stream>>>(xmap, wmap, perm, offsets, out, T, k, D,
                                                         E, De, status, wait_limit_ns);
    return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

// ------------------------------------------------- bounded-wait check kernel
__global__ void k_bounded_wait_probe(int32_t* status, uint64_t limit) {
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Nothing ever arrives on `bar`, so the wait can only end by its limit.
    if (threadIdx.x == 0 && !mbar_wait(smem_addr(&bar), 0, &abort, limit))
        report(status, PK_ERR_TIMEOUT);
}

cudaError_t launch_bounded_wait_probe(int32_t* status, uint64_t limit_ns, cudaStream_t stream) {
    k_bounded_wait_probe<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace pk
