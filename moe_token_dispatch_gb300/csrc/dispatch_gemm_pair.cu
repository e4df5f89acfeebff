// Token dispatch fused with the per-expert GEMM, CTA-pair form (sm_103a):
//   out[j, :] = x[perm[j] / k, :] @ W[e(j)]   for j in expert e's segment
// (the "token-dispatch + GEMM" of "Loads and Loads of Fluffy Kittens", "Key
// claims", Fig. 17), computed by 2-CTA clusters whose tensor-core operations
// span both SMs (tcgen05.mma.cta_group::2, M = 256, N = 256).
//
// Why a pair: in the one-CTA kernel each SM's ring carries 64 KiB per K-step
// (W tile 256 columns + two 128-row A tiles) and that ring, not the tensor
// core, bounds the GEMM. In a pair MMA each CTA supplies its own 128 rows of
// A and HALF of B's columns, and receives its 128 rows of D for all N columns.
// A unit here is (expert, two m-tiles, 512 columns): per K-step each CTA
// loads its 128 gathered rows (16 KiB) and its halves of two 256-column W
// blocks (2 x 16 KiB) -- 48 KiB per SM for the same tensor work that costs the
// one-CTA kernel 64 KiB, and the x rows of an expert are gathered 4 times
// (once per 512 columns) instead of 8.
//
// Per CTA, 11 warps, the roles of the one-CTA kernel:
//   warps 0-3   epilogue: the CTA's own 128 TMEM lanes (its own rows).
//   warp 4      TMEM owner in both CTAs (collective pair allocation); in
//               rank 0 one thread issues every MMA of the pair, after the
//               stage is full in both CTAs, and commits to both CTAs' barriers.
//   warp 5      W producer: TMA loads of this CTA's column halves.
//   warps 6,7,9,10  dispatch: cp.async gather of this CTA's 128 rows.
//   warp 8      in rank 1: relays "stage full" to rank 0 (a cp.async arrival
//               can only reach the CTA's own barrier). Idle in rank 0.
// Four 48 KiB stages. An expert's last m-tile pair may be half empty (odd
// number of m-tiles): the idle CTA still supplies its B halves; its rows are
// neither gathered nor stored.
//
// Measured on GB300 against the one-CTA kernel it is slower on every
// workload (ep 2.21 vs 1.79 ms, decode 1.36 vs 1.1 ms, FP8 ep 1.16 vs 1.00
// ms): both run at the latency of their ring, and every K-step here adds a
// cross-SM hop (relay to rank 0, multicast commit back) and waits for the
// slower of two SMs. It stays as an option behind pk_moe_set_gemm_kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pk_internal.h"
#include "pk_ptx.cuh"

namespace pk {
namespace dgp {

constexpr int BM = 128;                       // rows per CTA (half of the pair MMA's M)
constexpr int ROW_BYTES = 128;                // one 128-byte swizzle row per operand row per stage
constexpr int BOX = 64;                       // W box: 64 columns (bf16) or 64 rows (FP8)
constexpr int BOX_BYTES = BOX * ROW_BYTES;    // 8 KiB
constexpr int PAIR_N = 256;                   // N of one pair MMA
constexpr int HALF_N = PAIR_N / 2;            // B columns per CTA per pair MMA
constexpr int NBLK = 2;                       // pair-MMA column blocks per unit
constexpr int UNIT_N = PAIR_N * NBLK;         // 512 output columns per unit
constexpr int HALF_BYTES = HALF_N * ROW_BYTES;  // 16 KiB: one CTA's half of a block
constexpr int A_OFF = NBLK * HALF_BYTES;        // 32 KiB
constexpr int A_BYTES = BM * ROW_BYTES;         // 16 KiB
constexpr int STAGE_BYTES = A_OFF + A_BYTES;    // 48 KiB
constexpr int STAGES = 4;
constexpr uint32_t TMEM_COLS = 512;
constexpr int W_PREFETCH = 6;

constexpr int EPI_WARPS = 4;
constexpr int MMA_WARP = 4;
constexpr int W_WARP = 5;
constexpr int RELAY_WARP = 8;
constexpr int GATHER_THREADS = 128;
constexpr int THREADS = 11 * 32;
constexpr int ROWS_PER_PASS = GATHER_THREADS / 8;
constexpr int ROWS_PER_THREAD = BM / ROWS_PER_PASS;  // 8

__device__ __forceinline__ int gather_index(int warp, int lane) {
    if (warp == 6 || warp == 7) return (warp - 6) * 32 + lane;
    if (warp == 9 || warp == 10) return (warp - 7) * 32 + lane;
    return -1;
}

struct Ctrl {
    uint64_t full[STAGES];       // W arrive.expect_tx + one arrival per gather thread (own CTA)
    uint64_t peer_full[STAGES];  // rank 0 only: the relay's arrival for rank 1's stage
    uint64_t empty[STAGES];      // one pair commit
    uint64_t acc_full;           // one pair commit per unit
    uint64_t acc_empty;          // rank 0 only: 4 local + 4 remote epilogue warps
    uint64_t drain;              // final pair commit
    uint32_t tmem_base;
    int abort;
};

constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + static_cast<int>(sizeof(Ctrl)) + 64;

struct Unit {
    int e;
    int row0;      // first sorted row of the pair's two m-tiles
    int rows;      // valid rows of the pair (<= 256)
    int n0;        // first output column
    int nblk;      // 256-column blocks in this unit (1 or 2)
    bool shared_w; // other units of this expert read the same W tiles
};

struct Walker {
    const int32_t* off;
    int E, R, De, ntiles;
    int e;
    int64_t base;
    int lo, rows, groups;
    int64_t units;

    __device__ void init(const int32_t* o, int E_, int R_, int De_) {
        off = o; E = E_; R = R_; De = De_;
        ntiles = (De + UNIT_N - 1) / UNIT_N;
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
        groups = (rows + 2 * BM - 1) / (2 * BM);
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
        const int g = l / ntiles, n = l - g * ntiles;
        U.e = e;
        U.row0 = lo + g * 2 * BM;
        U.rows = min(2 * BM, rows - g * 2 * BM);
        U.n0 = n * UNIT_N;
        U.nblk = min(NBLK, (De - U.n0 + PAIR_N - 1) / PAIR_N);
        U.shared_w = groups > 1;
        return true;
    }
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                          uint64_t limit) {
    bool ok = true;
    if (lane_id() == 0) ok = mbar_wait(bar, parity, abort, limit);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}

// Records a timeout and stops both CTAs of the pair.
__device__ __forceinline__ void fail(volatile int* abort, uint32_t peer_abort, int32_t* status) {
    report(status, PK_ERR_TIMEOUT);
    *abort = 1;
    st_cluster_u32(peer_abort, 1u);
}

__device__ __forceinline__ void store_chunk(uint16_t* dst, const uint32_t (&v)[32], int col0,
                                            int De) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (col0 + g * 8 < De) {
            uint4 pkd;
            uint32_t* w = reinterpret_cast<uint32_t*>(&pkd);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[g * 8 + 2 * h]),
                                                          __uint_as_float(v[g * 8 + 2 * h + 1]));
                w[h] = *reinterpret_cast<uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(dst + col0 + g * 8) = pkd;
        }
    }
}

__device__ __forceinline__ void scale_chunk(uint32_t (&v)[32], int col0, int De, float rs,
                                            const float* __restrict__ sw_e) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (col0 + g * 8 < De) {
            const float4 s0 = __ldg(reinterpret_cast<const float4*>(sw_e + col0 + g * 8));
            const float4 s1 = __ldg(reinterpret_cast<const float4*>(sw_e + col0 + g * 8 + 4));
            const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int h = 0; h < 8; ++h)
                v[g * 8 + h] = __float_as_uint(__uint_as_float(v[g * 8 + h]) * rs * sc[h]);
        }
    }
}

template <bool kFp8>
__global__ void __launch_bounds__(THREADS, 1)
    k_dispatch_gemm_pair(const __grid_constant__ CUtensorMap wmap, const uint8_t* __restrict__ x,
                         const float* __restrict__ sx, const float* __restrict__ sw,
                         const int32_t* __restrict__ perm, const int32_t* __restrict__ offsets,
                         uint16_t* __restrict__ out, int32_t T, int32_t k, int32_t D, int32_t E,
                         int32_t De, int32_t* status, uint64_t limit) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    Ctrl* ctl = reinterpret_cast<Ctrl*>(smem_raw + (sbase - raw) + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int64_t pair = blockIdx.x >> 1;
    const int64_t npairs = gridDim.x >> 1;
    const int R = T * k;
    constexpr int ELEM = kFp8 ? 1 : 2;
    constexpr int BKE = ROW_BYTES / ELEM;   // K elements per stage
    constexpr int KCHUNK = 16 / ELEM;
    const int nk = (D + BKE - 1) / BKE;
    const int nb_count = (De + BOX - 1) / BOX;  // FP8 blocked W: 64-column blocks per expert

    const uint32_t full0 = smem_addr(&ctl->full[0]);
    const uint32_t peer_full0 = smem_addr(&ctl->peer_full[0]);
    const uint32_t empty0 = smem_addr(&ctl->empty[0]);
    const uint32_t acc_full = smem_addr(&ctl->acc_full);
    const uint32_t acc_empty = smem_addr(&ctl->acc_empty);
    const uint32_t drain = smem_addr(&ctl->drain);
    volatile int* abort = &ctl->abort;
    const uint32_t peer_abort = map_to_cta(smem_addr(&ctl->abort), rank ^ 1u);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1 + GATHER_THREADS);
            mbar_init(peer_full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * EPI_WARPS);
        mbar_init(drain, 1);
        ctl->abort = 0;
        fence_barrier_init();
    }
    if (warp == W_WARP && lane == 0) prefetch_tensormap(&wmap);
    if (warp == MMA_WARP) {
        tmem_alloc_pair(smem_addr(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised, TMEM allocated in both
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    const int gt = gather_index(warp, lane);
    if (gt >= 0) {
        // ------------------------------------------------------ dispatch
        const int c = gt & 7;
        const int rb = gt >> 3;
        const uint32_t swz = static_cast<uint32_t>((c ^ (rb & 7)) << 4);
        const uint64_t pol_x = policy_evict_last();
        Walker wk;
        wk.init(offsets, E, R, De);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true, bad = false;
        for (int64_t u = pair; ok; u += npairs) {
            Unit U;
            if (!wk.find(u, U)) break;
            const int my0 = static_cast<int>(rank) * BM;
            const int my_rows = max(0, min(BM, U.rows - my0));
            const char* src[ROWS_PER_THREAD];
#pragma unroll
            for (int i = 0; i < ROWS_PER_THREAD; ++i) {
                const int r = rb + ROWS_PER_PASS * i;
                const char* p = nullptr;
                if (r < my_rows) {
                    int f = __ldg(perm + U.row0 + my0 + r);
                    if (f < 0 || f >= R) {
                        bad = true;
                        f = 0;
                    }
                    p = reinterpret_cast<const char*>(x + static_cast<int64_t>(f / k) * D * ELEM) +
                        c * 16;
                }
                src[i] = p;
            }
            for (int ks = 0; ks < nk; ++ks) {
                if (!warp_wait(empty0 + 8 * stage, phase ^ 1u, abort, limit)) {
                    if (lane == 0) fail(abort, peer_abort, status);
                    ok = false;
                    break;
                }
                const uint32_t dst0 = sbase + stage * STAGE_BYTES + A_OFF + rb * 128 + swz;
                const uint32_t nbytes = (ks * BKE + c * KCHUNK < D) ? 16u : 0u;
                const int64_t koff = static_cast<int64_t>(ks) * ROW_BYTES;
#pragma unroll
                for (int i = 0; i < ROWS_PER_THREAD; ++i)
                    if (src[i])
                        cp_async_16(dst0 + i * (ROWS_PER_PASS * 128),
                                    nbytes ? src[i] + koff : src[i], nbytes, pol_x);
                cp_async_arrive_noinc(full0 + 8 * stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        cp_async_wait_all();
        if (bad) report(status, PK_ERR_BAD_INDEX);
    } else if (warp == W_WARP) {
        // ----------------------------------------------------- W producer
        if (lane == 0) {
            const uint64_t pol_once = policy_evict_first();
            const uint64_t pol_reuse = policy_evict_last();
            // first column of this CTA's half of block nb, box h
            auto col_of = [&](const Unit& U, int nb, int h) {
                return U.n0 + nb * PAIR_N + static_cast<int>(rank) * HALF_N + h * BOX;
            };
            auto load_box = [&](uint32_t dst, const Unit& U, int col, int ks, uint32_t bar,
                                uint64_t pol) {
                if (kFp8)
                    tma_load_2d(dst, &wmap, 0, ((U.e * nb_count + col / BOX) * nk + ks) * BOX, bar,
                                pol);
                else
                    tma_load_3d(dst, &wmap, col, ks * BKE, U.e, bar, pol);
            };
            auto prefetch_box = [&](const Unit& U, int col, int ks) {
                if (kFp8)
                    tma_prefetch_2d(&wmap, 0, ((U.e * nb_count + col / BOX) * nk + ks) * BOX);
                else
                    tma_prefetch_3d(&wmap, col, ks * BKE, U.e);
            };
            Walker wk, pf;
            wk.init(offsets, E, R, De);
            pf.init(offsets, E, R, De);
            int64_t pf_u = pair;
            int pf_ks = 0;
            Unit PU;
            bool pf_live = pf.find(pf_u, PU);
            auto prefetch_one = [&]() {
                if (!pf_live) return;
                for (int nb = 0; nb < PU.nblk; ++nb)
                    for (int h = 0; h < HALF_N / BOX; ++h) {
                        const int col = col_of(PU, nb, h);
                        if (col < De) prefetch_box(PU, col, pf_ks);
                    }
                if (++pf_ks == nk) {
                    pf_ks = 0;
                    pf_u += npairs;
                    pf_live = pf.find(pf_u, PU);
                }
            };
            for (int i = 0; i < W_PREFETCH; ++i) prefetch_one();
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0;
            bool ok = true;
            for (int64_t u = pair; ok; u += npairs) {
                Unit U;
                if (!wk.find(u, U)) break;
                const uint64_t pol = U.shared_w ? pol_reuse : pol_once;
                const uint32_t tx = static_cast<uint32_t>(U.nblk * HALF_BYTES);
                for (int ks = 0; ks < nk; ++ks) {
                    prefetch_one();
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort, limit)) {
                        fail(abort, peer_abort, status);
                        ok = false;
                        break;
                    }
                    const uint32_t full = full0 + 8 * stage;
                    mbar_arrive_expect_tx(full, tx);
                    const uint32_t sb = sbase + stage * STAGE_BYTES;
                    // boxes past D_expert read zeros (bf16) or unused codes (FP8):
                    // their output columns are never stored
                    for (int nb = 0; nb < U.nblk; ++nb)
                        for (int h = 0; h < HALF_N / BOX; ++h)
                            load_box(sb + nb * HALF_BYTES + h * BOX_BYTES, U, col_of(U, nb, h), ks,
                                     full, pol);
                    issued |= 1u << stage;
                    issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait(full0 + 8 * s, (issued_par >> s) & 1u, nullptr, limit);
        }
        __syncwarp();
    } else if (warp == RELAY_WARP) {
        // ------------------------------------- rank 1: stage-full relay
        if (rank == 1 && lane == 0) {
            const uint32_t leader_pf0 = map_to_cta(peer_full0, 0);
            Walker wk;
            wk.init(offsets, E, R, De);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int64_t u = pair; ok; u += npairs) {
                Unit U;
                if (!wk.find(u, U)) break;
                for (int ks = 0; ks < nk; ++ks) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort, limit)) {
                        fail(abort, peer_abort, status);
                        ok = false;
                        break;
                    }
                    // the gathered rows were written through the generic proxy
                    fence_proxy_async_smem();
                    mbar_arrive_remote(leader_pf0 + 8 * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ----------------------------------------------------------- MMA
        if (rank == 0 && lane == 0) {
            Walker wk;
            wk.init(offsets, E, R, De);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t idesc = kFp8 ? idesc_e4m3_f32(2 * BM, PAIR_N)
                                        : idesc_bf16_f32(2 * BM, PAIR_N, true);
            // A: K-major, rows 128 B apart, 8-row groups 1024 B apart.
            // B (bf16): MN-major, 64-column blocks 8 KiB apart, 8-row K groups
            // 1024 B apart; a K step of 16 rows is 2 KiB. B (FP8): K-major like A.
            const uint64_t a_desc0 = sdesc_sw128(sbase + A_OFF, 16, 1024);
            const uint64_t b_desc0 =
                kFp8 ? sdesc_sw128(sbase, 16, 1024) : sdesc_sw128(sbase, BOX_BYTES, 1024);
            constexpr uint32_t b_step = kFp8 ? (32 >> 4) : ((16 * 128) >> 4);
            for (int64_t u = pair; ok; u += npairs) {
                Unit U;
                if (!wk.find(u, U)) break;
                if (!mbar_wait_cluster(acc_empty, acc_phase ^ 1u, abort, limit)) {
                    fail(abort, peer_abort, status);
                    break;
                }
                tc_fence_after_sync();
                for (int ks = 0; ks < nk; ++ks) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort, limit) ||
                        !mbar_wait_cluster(peer_full0 + 8 * stage, phase, abort, limit)) {
                        fail(abort, peer_abort, status);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    fence_proxy_async_smem();
                    const uint64_t sdelta = static_cast<uint64_t>(stage) * (STAGE_BYTES >> 4);
                    const uint64_t a_st = a_desc0 + sdelta;
                    for (int nb = 0; nb < U.nblk; ++nb) {
                        const uint64_t b_st =
                            b_desc0 + sdelta + static_cast<uint64_t>(nb) * (HALF_BYTES >> 4);
                        const uint32_t d = tmem + static_cast<uint32_t>(nb * PAIR_N);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            if (kFp8)
                                mma_pair_f8(d, a_st + kk * (32 >> 4), b_st + kk * b_step, idesc,
                                            (ks | kk) != 0 ? 1u : 0u);
                            else
                                mma_pair_bf16(d, a_st + kk * (32 >> 4), b_st + kk * b_step, idesc,
                                              (ks | kk) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit_pair(empty0 + 8 * stage, 3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair(acc_full, 3);
                acc_phase ^= 1u;
            }
            mma_commit_pair(drain, 3);
        }
        // both CTAs: every MMA of the pair (which reads this CTA's shared
        // memory and writes its TMEM) has completed before either leaves
        if (lane == 0) mbar_wait(drain, 0, nullptr, limit);
        __syncwarp();
    } else if (warp < EPI_WARPS) {
        // ------------------------------------------------------ epilogue
        const int q = warp;
        const uint32_t acc_empty_leader = map_to_cta(acc_empty, 0);
        Walker wk;
        wk.init(offsets, E, R, De);
        uint32_t acc_phase = 0;
        for (int64_t u = pair;; u += npairs) {
            Unit U;
            if (!wk.find(u, U)) break;
            if (!warp_wait(acc_full, acc_phase, abort, limit)) {
                if (lane == 0) fail(abort, peer_abort, status);
                break;
            }
            tc_fence_after_sync();
            const int my0 = static_cast<int>(rank) * BM;
            const int my_rows = max(0, min(BM, U.rows - my0));
            const int r = q * 32 + lane;
            const bool valid = r < my_rows;
            const bool any = q * 32 < my_rows;  // warp-uniform
            uint16_t* orow = out + static_cast<int64_t>(U.row0 + my0 + r) * De;
            float rs = 1.0f;
            const float* sw_e = nullptr;
            if (kFp8) {
                if (valid) {
                    const int f = __ldg(perm + U.row0 + my0 + r);
                    rs = (f >= 0 && f < R) ? __ldg(sx + f / k) : 0.0f;
                }
                sw_e = sw + static_cast<int64_t>(U.e) * De;
            }
            const int nchunk = U.nblk * (PAIR_N / 32);
            bool released = false;
            if (any) {
                const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16);
                for (int cc = 0; cc < nchunk; cc += 2) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(tbase + cc * 32, v0);
                    tmem_ld_32x32b_x32(tbase + cc * 32 + 32, v1);
                    tmem_wait_ld();
                    if (cc + 2 >= nchunk) {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            if (rank == 0) mbar_arrive(acc_empty);
                            else mbar_arrive_remote(acc_empty_leader);
                        }
                        released = true;
                    }
                    const int col = U.n0 + cc * 32;
                    if (valid && col < De) {
                        if (kFp8) {
                            scale_chunk(v0, col, De, rs, sw_e);
                            scale_chunk(v1, col + 32, De, rs, sw_e);
                        }
                        store_chunk(orow, v0, col, De);
                        store_chunk(orow, v1, col + 32, De);
                    }
                }
            }
            if (!released) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0) mbar_arrive(acc_empty);
                    else mbar_arrive_remote(acc_empty_leader);
                }
            }
            acc_phase ^= 1u;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // neither CTA frees TMEM or leaves while its peer may still arrive on it
    if (warp == MMA_WARP) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

}  // namespace dgp

namespace {
std::mutex g_pair_mu;
int g_pair_clusters[64];  // 0: not yet queried
bool g_pair_attr[64];
}  // namespace

int launch_dispatch_gemm_pair(bool fp8, const void* x, const float* sx, const int32_t* perm,
                              const int32_t* offsets, const void* W, const float* sw, int32_t T,
                              int32_t k, int32_t D, int32_t E, int32_t De, uint16_t* out,
                              int32_t* status, cudaStream_t stream, uint64_t wait_limit_ns) {
    using namespace dgp;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PK_ERR_CUDA;
    auto kern = fp8 ? k_dispatch_gemm_pair<true> : k_dispatch_gemm_pair<false>;
    int clusters;
    {
        std::lock_guard<std::mutex> lk(g_pair_mu);
        if (!g_pair_attr[dev]) {
            if (cudaFuncSetAttribute(k_dispatch_gemm_pair<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SMEM_BYTES) != cudaSuccess ||
                cudaFuncSetAttribute(k_dispatch_gemm_pair<false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SMEM_BYTES) != cudaSuccess)
                return PK_ERR_CUDA;
            g_pair_attr[dev] = true;
        }
        if (g_pair_clusters[dev] == 0) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            int sms = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return PK_ERR_CUDA;
            cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
            cfg.blockDim = dim3(THREADS, 1, 1);
            cfg.dynamicSmemBytes = SMEM_BYTES;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, k_dispatch_gemm_pair<false>, &cfg) !=
                    cudaSuccess ||
                n < 1)
                return PK_ERR_UNSUPPORTED;
            g_pair_clusters[dev] = n < sms / 2 ? n : sms / 2;
        }
        clusters = g_pair_clusters[dev];
    }
    CUtensorMap wmap;
    const int rc = make_w_map(fp8, W, D, E, De, &wmap);
    if (rc != PK_OK) return rc;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint8_t* x8 = static_cast<const uint8_t*>(x);
    cudaError_t err = cudaLaunchKernelEx(&cfg, kern, wmap, x8, sx, sw, perm, offsets, out, T, k, D,
                                         E, De, status, wait_limit_ns);
    return err == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

}  // namespace pk
