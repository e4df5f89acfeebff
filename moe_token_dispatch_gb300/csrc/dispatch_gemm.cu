// Token dispatch fused with the per-expert up-projection GEMM on sm_103a:
//   out[j, :] = x[perm[j] / k, :] @ W[e(j)]   for j in expert e's segment
// -- the "token-dispatch + GEMM" of "Loads and Loads of Fluffy Kittens"
// ("Key claims", Fig. 17) on one device. What carries over from the pages is
// their intra-SM overlap (section "Using the Right Overlapping Schedule"):
// producer warps move tiles while the tensor cores stay busy.
//
// Persistent kernel, one CTA per SM, 12 warps:
//   warps 0-3  epilogue: tcgen05.ld of the warp's TMEM lane quarter, bf16
//              round-to-nearest-even, stores of the valid rows and columns
//              (32-byte stores of eight rows x 128 B after a transpose inside
//              each group of four lanes); between units the warps sleep
//              between tests of the accumulator barrier.
//   warp 4     MMA issuer (one thread) and TMEM owner: tcgen05.mma M=128 x
//              N=bn x K=16 per m-tile (M=64 for a last m-tile of at most 64
//              rows) into fp32 accumulators in TMEM; each commit frees a
//              shared-memory slot or hands the unit's accumulators to the
//              epilogue.
//   warp 5     W producer (one thread): per K-step of 64 rows, TMA-loads the
//              W_e tile [64 x bn] as 64x64 boxes, 128-byte swizzle (MN-major
//              operand).
//   warps 6,7,9,10  dispatch: gather the routed x rows of the unit's m-tiles
//              0 and 1 with 16-byte cp.async into K-major 128-byte-swizzled
//              tiles (each warp instruction moves four whole 128-byte row
//              segments); each thread's copies arrive on the K-step's full
//              barrier when they land, and the MMA thread fences them into the
//              async proxy after its wait, before the tensor cores read them.
//   warp 11    dispatch of m-tile 2 of 3-m-tile units, the same way.
//   warp 8     scheduler: walks this CTA's units 32 experts at a time (one
//              expert per lane) and queues each unit's shape in shared memory
//              (eight entries, full/empty barriers), so no other role walks
//              the expert offsets. Warps share an SM sub-partition with the
//              warps whose index is equal mod 4; this keeps the busy gather
//              warps off the MMA issuer's sub-partition.
// Two rings of shared-memory slots connect producers and MMA: W slots and
// A slots (m-tiles 0 and 1) of 32 KiB, one of each per K-step; a 3-m-tile
// unit puts its m-tile 2 in the second half of its W slot (its W tile is
// 16 KiB). When x is larger than L2 can keep beside the W stream, some
// gathered rows come from DRAM, and the A ring needs the depth: three W and
// four A slots (measured on ep: one A slot less costs 31 %, one W slot less
// nothing). When x stays in L2, four W and three A slots hide more of the W
// stream's HBM latency (decode, mid: 1.4-6 % faster). One full and one
// empty barrier per K-step (a ring of eight pairs, indexed by K-step)
// serve both rings: the full barrier counts the W bytes and every gather
// thread's arrival, so the MMA thread waits once per K-step, and its one
// commit frees both slots; each producer waits for the K-step that last used
// its slot. m-tile 2 has a warp of its own because a thread's cp.async
// arrivals cover all its earlier copies: with the shorter lead of the W slot
// it would hold back the arrivals of m-tiles 0 and 1.
//
// The same kernel, instantiated with kGather = false, is the grouped GEMM of
// rows that are already in expert order (the down-projection that follows the
// expert MLP: out2[j, :] = h[j, :] @ W2[e(j)]): each m-tile of A arrives by
// TMA as one 128-row box, m-tiles 0 and 1 from an A producer of their own
// (warp 6, lane 0) and m-tile 2 with W, and the other gather warps idle (with
// kFp8 too: E4M3 codes of h with one scale per row). It always runs four W
// and three A slots: an expert's A rows are re-read by its concurrent n-tiles
// from L2, and the W stream gains the deeper ring (ep 1.683 -> 1.604 ms).
//
// With kFp8, the same pipeline is the FP8 variant of the expert GEMM: x and W
// arrive as E4M3 codes with one fp32 scale per token row and per (expert,
// output column); a stage then holds K = 128 codes (still 128 bytes per row),
// W is read K-major from a blocked layout in which each 64-column x 128-code
// box is one contiguous 8 KiB block (so every TMA box is a single contiguous
// read from HBM), the MMAs are tcgen05.mma kind::f8f6f4 with K = 32, and the
// epilogue multiplies each accumulator by its row's and column's scale (both
// loaded into registers while the unit's MMAs still run, so that the
// accumulators are not held in TMEM across those loads).
//
// With kMx (and kFp8) the codes carry one E8M0 scale per 32 elements along D
// (MXFP8): units of at most two m-tiles and 192 columns, so that four
// 16-column scale buffers fit in TMEM beside the accumulators; each K-step's
// W scale piece follows its codes in the W slot, warp 11 gathers the rows'
// scale bytes into the same slot, and the MMA thread copies both into TMEM
// (tcgen05.cp) before the block-scaled MMAs (kind::mxf8f6f4).
//
// Work unit = (expert e, group of m-tiles, n-tile), with a shape chosen per
// expert so that TMEM (512 fp32 columns x 128 lanes) holds every accumulator
// of the unit and each W tile is loaded once per unit:
//   <= 2 m-tiles (<= 256 rows): one group, n-tiles of 256 columns;
//   3 m-tiles (257..384 rows):  one group of three, n-tiles of 128 columns;
//   >= 4 m-tiles:               groups of two, n-tiles of 256 columns.
// So an expert with at most 384 rows streams W_e from memory exactly once.
// Units are numbered expert by expert, group-major then n-tile, and dealt
// round-robin to the CTAs: the n-tiles of one row group (which gather the same
// rows) run side by side, and the groups of a heavy expert reuse W_e from L2
// (its W loads are marked evict-last; single-group experts mark W
// evict-first, as each tile is needed once). Experts with no rows add no
// units.
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
constexpr int ROW_BYTES = 128;               // bytes of one row segment per stage (either type)
constexpr int B_BOX = 64;                    // W box: 64 columns (bf16) or 64 rows (FP8 codes)
constexpr int B_BOX_BYTES = B_BOX * ROW_BYTES;  // 8 KiB
constexpr int A_BYTES = BM * BK * 2;         // 16 KiB per m-tile
// Two rings, one slot per K-step each, seven 32 KiB slots in all: a W slot
// holds the W tile (bn_max x 128 B; 3-m-tile units, bn_max = 128, put their
// third A tile in its second half), an A slot m-tiles 0 and 1. The split is
// a template parameter (kWDeep): three W + four A slots when the gathered
// rows may miss L2 (x larger than L2 can keep beside the W stream: their
// DRAM-latency tail needs the deeper A ring), four W + three A slots when x
// stays in L2, so that the W ring hides more of HBM's latency.
constexpr int SLOTS = 7;
constexpr int W_SLOT = 32 * 1024;
constexpr int A_SLOT = 2 * A_BYTES;
static_assert(W_SLOT == A_SLOT, "one slot size for both rings");
constexpr int RING_BYTES = SLOTS * W_SLOT;   // 224 KiB
// x sizes (bytes) up to which the deep W ring is used
constexpr int64_t DEEP_W_MAX_X_BYTES = int64_t{24} << 20;
// K-step j uses full/empty barrier pair j mod NBAR. Each producer waits for
// the K-step its slot's previous user ran (j - W slots for a W slot and for
// m-tile 2 of a 3-m-tile unit, which lives in the W slot's second half;
// j - A slots for an A slot) before it arrives for K-step j. With more
// barrier pairs than either lag, the phase a producer waits for can never be
// overtaken by the next phase of the same barrier, and no arrival can reach
// a barrier whose previous phase is still open.
constexpr int NBAR = 8;
constexpr int UMMA_K = 16;
// A unit whose last m-tile holds at most 64 rows issues that m-tile's MMAs
// with M = 64 (bf16 and FP8; not MX). An M = 64 MMA takes the tensor core as
// long as an M = 128 one but does half the multiplies: on the power-capped
// GB300 the saved energy raises the clock (ep: the 3-m-tile experts' third
// m-tile holds ~13 of 128 rows). Its accumulator rows 16 q .. 16 q + 15 sit
// in TMEM lanes 32 q .. 32 q + 15 (lane quarter q).
constexpr int BM_HALF = 64;
__device__ __forceinline__ bool half_last(int mpu, int rows) {
    return rows - (mpu - 1) * BM <= BM_HALF;
}
// MXFP8 (kMx): units of at most two m-tiles and 192 columns, so that the
// accumulators (384 TMEM columns) leave room for four 16-column buffers of
// block scales (one per A slot); each K-step's scales travel in the W slot
// after its 24 KiB of codes: W's (two 512-byte halves, 1 KiB) then the rows'
// (512 bytes per m-tile).
constexpr int MX_BN = 192;
constexpr int MX_SFB_OFF = MX_BN * ROW_BYTES;        // 24 KiB into the W slot
constexpr int MX_SFA_OFF = MX_SFB_OFF + 1024;
constexpr uint32_t MX_SF_TMEM = 2 * MX_BN;           // first scale column in TMEM
constexpr uint32_t MX_SF_COLS = 16;                  // per buffer: A m-tiles 0, 1, B halves
static_assert(MX_SFA_OFF + 2 * 512 <= W_SLOT, "MX scales fit the W slot");
constexpr uint32_t TMEM_COLS = 512;

constexpr int EPI_WARPS = 4;                 // warps 0..3
constexpr int MMA_WARP = 4;
constexpr int W_WARP = 5;
constexpr int GATHER_WARPS = 4;              // warps 6, 7, 9, 10: m-tiles 0 and 1
constexpr int GATHER_THREADS = GATHER_WARPS * 32;
constexpr int GATHER2_WARP = 11;             // m-tile 2 of 3-m-tile units
constexpr int THREADS = 12 * 32;

// Gather-thread index 0..127 of a thread in warps 6, 7, 9, 10; -1 otherwise.
__device__ __forceinline__ int gather_index(int warp, int lane) {
    if (warp == 6 || warp == 7) return (warp - 6) * 32 + lane;
    if (warp == 9 || warp == 10) return (warp - 7) * 32 + lane;
    return -1;
}
constexpr int ROWS_PER_PASS = GATHER_THREADS / 8;    // 8 threads per 128-byte row segment
constexpr int ROWS_PER_THREAD = BM / ROWS_PER_PASS;  // per m-tile
constexpr int MAX_MPU = 3;                   // m-tiles per unit
constexpr int ROWS2_PER_THREAD = BM / 4;     // warp 11: 4 rows per pass
constexpr int SCHED_WARP = 8;
constexpr int NQ = 8;                        // unit queue depth
constexpr int QWORDS = 8;                    // e, row0, rows, mpu, n0, bn, bn_max, shared_w
struct Ctrl {
    // One pair of barriers per K-step covers both rings: the K-step's W slot
    // and A slot fill up together and are freed by the same commit.
    uint64_t wfull[NBAR];       // W producer arrive + tx bytes (+ one arrival per gather thread)
    uint64_t wempty[NBAR];      // one tcgen05.commit
    uint64_t acc_full;          // one tcgen05.commit per unit
    uint64_t acc_empty;         // one arrive per epilogue warp
    uint64_t drain;
    uint64_t qfull[NQ];         // scheduler arrive
    uint64_t qempty[NQ];        // one arrive per consumer (thread or warp)
    int q[NQ][QWORDS];
    uint32_t tmem_base;
    int abort;
};

constexpr int SMEM_BYTES = RING_BYTES + 1024 + static_cast<int>(sizeof(Ctrl)) + 64;
static_assert(SMEM_BYTES <= 232448, "shared memory per block");

// Slot index and phase parity of one ring, advanced once per K-step.
template <int N>
struct Cursor {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next() {
        if (++s == N) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Cursor over the barrier ring that trails the current K-step by L: entry
// (j - L) mod NBAR and the parity of that K-step's phase. Its first L
// positions name phase -1 (parity 1), which a fresh barrier reports
// complete, so the first fills of a ring do not wait.
template <int L>
__device__ __forceinline__ Cursor<NBAR> lag_cursor() {
    Cursor<NBAR> c;
    c.s = (NBAR - L) % NBAR;
    c.ph = 1u;
    return c;
}

struct Unit {
    int e;        // expert
    int row0;     // first sorted row of the unit
    int rows;     // valid rows
    int mpu;      // m-tiles in this unit
    int n0;       // first output column
    int bn;       // n-tile width (a multiple of 64)
    int bn_max;   // n-tile width of this expert's units: accumulator column stride
    bool shared_w;  // other units of this expert load the same W tiles
};

// Sleep between tests of a wait that spans a whole unit (epilogue, scheduler).
constexpr uint32_t IDLE_SLEEP_NS = 1024;

// One lane waits; the warp learns the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                          uint64_t limit) {
    bool ok = true;
    if (lane_id() == 0) ok = mbar_wait(bar, parity, abort, limit);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}

// Next unit from the scheduler's queue: 1 = a unit, 0 = no more units,
// -1 = the wait gave up (abort or time limit). kWarp: every lane of the
// warp calls this and lane 0 does the barrier traffic.
template <bool kWarp>
__device__ __forceinline__ int q_pop(uint32_t qfull0, uint32_t qempty0, const int (*q)[QWORDS],
                                     Cursor<NQ>& qc, Unit& U, const volatile int* abort,
                                     uint64_t limit) {
    const bool ok = kWarp ? warp_wait(qfull0 + 8 * qc.s, qc.ph, abort, limit)
                          : mbar_wait(qfull0 + 8 * qc.s, qc.ph, abort, limit);
    if (!ok) return -1;
    const volatile int* d = q[qc.s];
    U.e = d[0]; U.row0 = d[1]; U.rows = d[2]; U.mpu = d[3];
    U.n0 = d[4]; U.bn = d[5]; U.bn_max = d[6]; U.shared_w = d[7] != 0;
    if (kWarp) {
        __syncwarp();
        if (lane_id() == 0) mbar_arrive(qempty0 + 8 * qc.s);
    } else {
        mbar_arrive(qempty0 + 8 * qc.s);
    }
    qc.next();
    return U.e >= 0 ? 1 : 0;
}

__device__ __forceinline__ void fail(volatile int* abort, int32_t* status) {
    report(status, PK_ERR_TIMEOUT);
    *abort = 1;
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
    __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t*>(&b2);
}

// 32 fp32 accumulators of one row -> bf16 columns [col0, col0 + 32), those
// below De. wide: 32-byte stores (row and column offsets 32-byte aligned),
// so a warp's store instruction writes 32 whole sectors, else 16-byte ones.
__device__ __forceinline__ void store_row_chunk(uint16_t* dst, const uint32_t (&v)[32], int col0,
                                                int De, bool wide) {
    if (wide) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            if (col0 + g * 16 < De) {
                uint32_t w[8];
#pragma unroll
                for (int h = 0; h < 8; ++h) w[h] = pack_bf16x2(v[g * 16 + 2 * h], v[g * 16 + 2 * h + 1]);
                asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(
                                 dst + col0 + g * 16),
                             "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                             "r"(w[6]), "r"(w[7])
                             : "memory");
            }
        }
        return;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (col0 + g * 8 < De) {
            uint4 pkd;
            pkd.x = pack_bf16x2(v[g * 8 + 0], v[g * 8 + 1]);
            pkd.y = pack_bf16x2(v[g * 8 + 2], v[g * 8 + 3]);
            pkd.z = pack_bf16x2(v[g * 8 + 4], v[g * 8 + 5]);
            pkd.w = pack_bf16x2(v[g * 8 + 6], v[g * 8 + 7]);
            *reinterpret_cast<uint4*>(dst + col0 + g * 8) = pkd;
        }
    }
}

// 64 accumulator columns of the warp's 32 rows (lane = row; v0 holds columns
// col0 .. col0+31, v1 the next 32) -> bf16, then a 4 x 4 transpose of 32-byte
// blocks inside each group of four lanes, so that lane 4g + c holds block c
// (16 columns) of rows 4g .. 4g+3 and each of the four store instructions
// writes eight rows x 128 contiguous bytes (instead of 32 rows x 32 bytes).
// Every lane of the warp must call this; rows >= nrows and columns >= De are
// not stored. Needs De % 16 == 0 and a 32-byte aligned out.
__device__ __forceinline__ void store_rows_quad(uint16_t* out, int64_t row0, int nrows, int De,
                                                const uint32_t (&v0)[32], const uint32_t (&v1)[32],
                                                int col0) {
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int c = lane & 3;
    uint32_t b0[8], b1[8], b2[8], b3[8];  // 16-column blocks 0..3 of this lane's row
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        b0[w] = pack_bf16x2(v0[2 * w], v0[2 * w + 1]);
        b1[w] = pack_bf16x2(v0[16 + 2 * w], v0[16 + 2 * w + 1]);
        b2[w] = pack_bf16x2(v1[2 * w], v1[2 * w + 1]);
        b3[w] = pack_bf16x2(v1[16 + 2 * w], v1[16 + 2 * w + 1]);
    }
    const bool odd = (c & 1) != 0, hi = (c & 2) != 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        // lanes 2a, 2a+1 swap across blocks (0,1) and (2,3)
        uint32_t r = __shfl_xor_sync(0xffffffffu, odd ? b0[w] : b1[w], 1);
        if (odd) b0[w] = r; else b1[w] = r;
        r = __shfl_xor_sync(0xffffffffu, odd ? b2[w] : b3[w], 1);
        if (odd) b2[w] = r; else b3[w] = r;
        // lanes a, a+2 swap across block pairs (0,1) and (2,3)
        r = __shfl_xor_sync(0xffffffffu, hi ? b0[w] : b2[w], 2);
        if (hi) b0[w] = r; else b2[w] = r;
        r = __shfl_xor_sync(0xffffffffu, hi ? b1[w] : b3[w], 2);
        if (hi) b1[w] = r; else b3[w] = r;
    }
    const int col = col0 + 16 * c;
    if (col >= De) return;
    const int rq = lane & ~3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (rq + i >= nrows) break;
        const uint32_t* s = i == 0 ? b0 : i == 1 ? b1 : i == 2 ? b2 : b3;
        uint16_t* dst = out + (row0 + rq + i) * static_cast<int64_t>(De) + col;
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(s[0]),
                     "r"(s[1]), "r"(s[2]), "r"(s[3]), "r"(s[4]), "r"(s[5]), "r"(s[6]), "r"(s[7])
                     : "memory");
    }
}

// FP8 epilogue: accumulator x row scale, then x column scale (fp32). Lane L
// holds the scale of column col0 + L (`cs`); column j's is broadcast to the
// whole warp by a shuffle, so every lane of the warp must call this.
__device__ __forceinline__ void scale_chunk(uint32_t (&v)[32], float rs, float cs) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
        v[j] = __float_as_uint((__uint_as_float(v[j]) * rs) * __shfl_sync(0xffffffffu, cs, j));
}

// kMx (with kGather and kFp8): E4M3 codes with one E8M0 scale per 32 codes
// along D: sx_ is the rows' scale bytes [T, D / 32], sw_ the weights' scale
// pieces (1 KiB per 192-column tile and K-step); otherwise (FP8) both are
// fp32 scales [T] and [E, De].
template <bool kGather, bool kFp8, bool kMx = false, bool kWDeep = false>
__global__ void __launch_bounds__(THREADS, 1)
    k_dispatch_gemm(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap amap,
                    const uint8_t* __restrict__ x, const void* __restrict__ sx_,
                    const void* __restrict__ sw_,
                    const int32_t* __restrict__ perm, const int32_t* __restrict__ offsets,
                    uint16_t* __restrict__ out, int32_t T, int32_t k, int32_t D, int32_t E,
                    int32_t De, int32_t* status, uint64_t limit, int64_t stall) {
    static_assert(!kMx || (kGather && kFp8), "MXFP8 is a form of the FP8 dispatch GEMM");
    constexpr int WS = kWDeep ? 4 : 3;        // W slots
    constexpr int AS = SLOTS - WS;            // A slots
    constexpr int A_RING = WS * W_SLOT;       // the A ring follows the W ring
    static_assert(NBAR > WS && NBAR > AS, "barrier ring shorter than a slot lag");
    // Grouped GEMM (rows already in expert order, A by TMA) with the deep W
    // ring: the W producer can no longer load A too (it waits for its W
    // slot's previous user, WS K-steps back, but an A slot's previous user is
    // only AS < WS back), so an A producer of its own (warp 6, lane 0) loads
    // m-tiles 0 and 1; the W producer loads W and m-tile 2, which lives in
    // the W slot.
    constexpr bool kSplitA = !kGather && kWDeep;
    const float* sx = static_cast<const float*>(sx_);
    const float* sw = static_cast<const float*>(sw_);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (sbase - raw);
    Ctrl* ctl = reinterpret_cast<Ctrl*>(base_ptr + RING_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int R = T * k;
    constexpr int ELEM = kFp8 ? 1 : 2;              // bytes per element
    constexpr int BKE = ROW_BYTES / ELEM;           // K elements per K-step
    constexpr int KCHUNK = 16 / ELEM;               // K elements per 16-byte chunk
    const int nk = (D + BKE - 1) / BKE;
    // FP8 blocked W: box (e, column block nb, K block kb) starts at row
    // ((e * NB + nb) * nk + kb) * 64 of the [rows, 128] code matrix.
    const int nb_count = (De + B_BOX - 1) / B_BOX;
    auto fp8_box_row = [&](int e, int nb, int kb) {
        return ((e * nb_count + nb) * nk + kb) * B_BOX;
    };
    // shared-memory address of m-tile mt of a K-step using W slot ws, A slot as
    auto a_tile = [&](int ws, int as, int mt) -> uint32_t {
        return mt < 2 ? sbase + A_RING + as * A_SLOT + mt * A_BYTES
                      : sbase + ws * W_SLOT + (W_SLOT - A_BYTES);
    };

    const uint32_t wfull0 = smem_addr(&ctl->wfull[0]);
    const uint32_t wempty0 = smem_addr(&ctl->wempty[0]);
    const uint32_t acc_full = smem_addr(&ctl->acc_full);
    const uint32_t acc_empty = smem_addr(&ctl->acc_empty);
    const uint32_t drain = smem_addr(&ctl->drain);
    const uint32_t qfull0 = smem_addr(&ctl->qfull[0]);
    const uint32_t qempty0 = smem_addr(&ctl->qempty[0]);
    volatile int* abort = &ctl->abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NBAR; ++s) {
            mbar_init(wfull0 + 8 * s, kGather ? 1 + GATHER_THREADS + 32 : (kSplitA ? 2 : 1));
            mbar_init(wempty0 + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, EPI_WARPS);
        mbar_init(drain, 1);
        for (int s = 0; s < NQ; ++s) {
            mbar_init(qfull0 + 8 * s, 1);
            mbar_init(qempty0 + 8 * s,
                      (kGather ? GATHER_WARPS + 1 : 0) + (kSplitA ? 1 : 0) + 2 + EPI_WARPS);
        }
        ctl->abort = 0;
        fence_barrier_init();
    }
    if (warp == W_WARP && lane == 0) {
        prefetch_tensormap(&wmap);
        if (!kGather) prefetch_tensormap(&amap);
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_addr(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    // Without kGather the rows arrive by TMA (W producer) and warps 6, 7, 9,
    // 10 fall through to the final barrier.
    const int gt = gather_index(warp, lane);
    if (kGather && gt >= 0) {
        // ---------------------------------------- dispatch, m-tiles 0 and 1
        const int c = gt & 7;          // 16-byte chunk of the 128-byte row segment
        const int rb = gt >> 3;        // first row of this thread (0..15)
        const uint32_t swz = static_cast<uint32_t>(((c ^ (rb & 7)) << 4));
        const uint64_t pol_x = policy_evict_last();  // rows are re-read by the unit's other n-tiles
        Cursor<NQ> qc;
        Cursor<NBAR> bc;
        Cursor<AS> ac;
        Cursor<NBAR> back = lag_cursor<AS>();  // the A slot's previous user
        bool ok = true, bad = false;
        while (ok) {
            Unit U;
            const int got = q_pop<true>(qfull0, qempty0, ctl->q, qc, U, abort, limit);
            if (got <= 0) {
                if (got < 0 && lane == 0) fail(abort, status);
                break;
            }
            const char* src[2][ROWS_PER_THREAD];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int i = 0; i < ROWS_PER_THREAD; ++i) {
                    const int r = mt * BM + rb + ROWS_PER_PASS * i;
                    const char* p = nullptr;
                    if (mt < U.mpu && r < U.rows) {
                        int f = __ldg(perm + U.row0 + r);
                        if (f < 0 || f >= R) {
                            bad = true;
                            f = 0;
                        }
                        p = reinterpret_cast<const char*>(x + static_cast<int64_t>(f / k) * D * ELEM) +
                            c * 16;
                    }
                    src[mt][i] = p;
                }
            for (int ks = 0; ks < nk; ++ks) {
                if (!warp_wait(wempty0 + 8 * back.s, back.ph, abort, limit)) {
                    if (lane == 0) fail(abort, status);
                    ok = false;
                    break;
                }
                const uint32_t nbytes = (ks * BKE + c * KCHUNK < D) ? 16u : 0u;
                const int64_t koff = static_cast<int64_t>(ks) * ROW_BYTES;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const uint32_t dst0 = sbase + A_RING + ac.s * A_SLOT + mt * A_BYTES + rb * 128 + swz;
#pragma unroll
                    for (int i = 0; i < ROWS_PER_THREAD; ++i)
                        if (src[mt][i])
                            cp_async_16(dst0 + i * (ROWS_PER_PASS * 128),
                                        nbytes ? src[mt][i] + koff : src[mt][i], nbytes, pol_x);
                }
                cp_async_arrive_noinc(wfull0 + 8 * bc.s);
                bc.next();
                ac.next();
                back.next();
            }
        }
        // Copies still in flight must land before the CTA may exit.
        cp_async_wait_all();
        if (bad) report(status, PK_ERR_BAD_INDEX);
    } else if (kMx && warp == GATHER2_WARP) {
        // --------------------------- MX: the rows' block scales, per K-step
        // Four scale bytes (the K-step's four 32-code blocks) of each row's
        // token, into the W slot as the 32-row x 16-byte pieces that
        // tcgen05.cp copies: row r of m-tile mt at byte (r % 32) * 16 +
        // (r / 32 % 4) * 4 of piece mt. Lane l takes rows l + 32 i.
        const uint8_t* sxm = static_cast<const uint8_t*>(sx_);
        const int nbr = D / 32;                   // scale bytes per token row
        Cursor<NQ> qc;
        Cursor<NBAR> bc;
        Cursor<WS> wc;
        Cursor<NBAR> back = lag_cursor<WS>();  // the W slot's previous user
        bool ok = true, bad = false;
        while (ok) {
            Unit U;
            const int got = q_pop<true>(qfull0, qempty0, ctl->q, qc, U, abort, limit);
            if (got <= 0) {
                if (got < 0 && lane == 0) fail(abort, status);
                break;
            }
            int tok[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = lane + 32 * i;
                int t = -1;
                if (r < U.rows) {
                    int f = __ldg(perm + U.row0 + r);
                    if (f < 0 || f >= R) {
                        bad = true;
                        f = 0;
                    }
                    t = f / k;
                }
                tok[i] = t;
            }
            for (int ks = 0; ks < nk; ++ks) {
                if (!warp_wait(wempty0 + 8 * back.s, back.ph, abort, limit)) {
                    if (lane == 0) fail(abort, status);
                    ok = false;
                    break;
                }
                const uint32_t dst0 = sbase + wc.s * W_SLOT + MX_SFA_OFF + lane * 16;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (tok[i] >= 0)
                        cp_async_4(dst0 + (i >> 2) * 512 + (i & 3) * 4,
                                   sxm + static_cast<int64_t>(tok[i]) * nbr + 4 * ks);
                cp_async_arrive_noinc(wfull0 + 8 * bc.s);
                bc.next();
                wc.next();
                back.next();
            }
        }
        cp_async_wait_all();
        if (bad) report(status, PK_ERR_BAD_INDEX);
    } else if (kGather && warp == GATHER2_WARP) {
        // -------------------------- dispatch, m-tile 2 of 3-m-tile units
        // Its own warp, so that its shorter lead (it writes the W slot's
        // second half, whose previous user is WS K-steps back) does not
        // hold back the arrivals of m-tiles 0 and 1, which a thread's
        // cp.async arrivals would otherwise cover together. Every K-step it
        // waits and arrives, also without rows to copy.
        const int c = lane & 7;
        const int rb = lane >> 3;      // rows rb + 4 i
        const uint64_t pol_x = policy_evict_last();
        Cursor<NQ> qc;
        Cursor<NBAR> bc;
        Cursor<WS> wc;
        Cursor<NBAR> back = lag_cursor<WS>();  // the W slot's previous user
        bool ok = true, bad = false;
        while (ok) {
            Unit U;
            const int got = q_pop<true>(qfull0, qempty0, ctl->q, qc, U, abort, limit);
            if (got <= 0) {
                if (got < 0 && lane == 0) fail(abort, status);
                break;
            }
            const int rows2 = U.mpu == 3 ? U.rows - 2 * BM : 0;  // valid rows of m-tile 2
            int tok[ROWS2_PER_THREAD];                            // element offset of each row's x
#pragma unroll
            for (int i = 0; i < ROWS2_PER_THREAD; ++i) {
                const int r = rb + 4 * i;
                int off = -1;
                if (r < rows2) {
                    int f = __ldg(perm + U.row0 + 2 * BM + r);
                    if (f < 0 || f >= R) {
                        bad = true;
                        f = 0;
                    }
                    off = f / k;
                }
                tok[i] = off;
            }
            for (int ks = 0; ks < nk; ++ks) {
                if (!warp_wait(wempty0 + 8 * back.s, back.ph, abort, limit)) {
                    if (lane == 0) fail(abort, status);
                    ok = false;
                    break;
                }
                if (rows2 > 0) {
                    const uint32_t nbytes = (ks * BKE + c * KCHUNK < D) ? 16u : 0u;
                    const int64_t koff = static_cast<int64_t>(ks) * ROW_BYTES;
                    const uint32_t dst0 = sbase + wc.s * W_SLOT + (W_SLOT - A_BYTES);
#pragma unroll
                    for (int i = 0; i < ROWS2_PER_THREAD; ++i) {
                        const int r = rb + 4 * i;
                        if (tok[i] >= 0) {
                            const char* p = reinterpret_cast<const char*>(
                                                x + static_cast<int64_t>(tok[i]) * D * ELEM) + c * 16;
                            cp_async_16(dst0 + r * 128 + static_cast<uint32_t>((c ^ (r & 7)) << 4),
                                        nbytes ? p + koff : p, nbytes, pol_x);
                        }
                    }
                }
                cp_async_arrive_noinc(wfull0 + 8 * bc.s);
                bc.next();
                wc.next();
                back.next();
            }
        }
        cp_async_wait_all();
        if (bad) report(status, PK_ERR_BAD_INDEX);
    } else if (kSplitA && warp == 6) {
        // ---------------------------- A producer (grouped GEMM, deep W ring)
        if (lane == 0) {
            const uint64_t pol_reuse = policy_evict_last();  // re-read by every n-tile
            Cursor<NQ> qc;
            Cursor<NBAR> bc;
            Cursor<AS> ac;
            Cursor<NBAR> back = lag_cursor<AS>();  // the A slot's previous user
            uint32_t a_issued = 0, a_par = 0;
            bool ok = true;
            while (ok) {
                Unit U;
                const int got = q_pop<false>(qfull0, qempty0, ctl->q, qc, U, abort, limit);
                if (got <= 0) {
                    if (got < 0) fail(abort, status);
                    break;
                }
                const int a_lo = U.mpu < 2 ? U.mpu : 2;
                for (int ks = 0; ks < nk; ++ks) {
                    if (!mbar_wait(wempty0 + 8 * back.s, back.ph, abort, limit)) {
                        fail(abort, status);
                        ok = false;
                        break;
                    }
                    const uint32_t full = wfull0 + 8 * bc.s;
                    mbar_arrive_expect_tx(full, static_cast<uint32_t>(a_lo * A_BYTES));
                    // rows past the expert's end are loaded but never stored
                    for (int mt = 0; mt < a_lo; ++mt)
                        tma_load_2d(sbase + A_RING + ac.s * A_SLOT + mt * A_BYTES, &amap, ks * BKE,
                                    U.row0 + mt * BM, full, pol_reuse);
                    a_issued |= 1u << bc.s;
                    a_par = (a_par & ~(1u << bc.s)) | (bc.ph << bc.s);
                    bc.next();
                    ac.next();
                    back.next();
                }
            }
            // Every copy this thread started must land before the CTA may exit
            // (after an abort a barrier may lack the W producer's bytes: the
            // first wait that runs out ends the drain, the copies have landed
            // long before).
            bool drained = true;
            for (int s = 0; s < NBAR && drained; ++s)
                if ((a_issued >> s) & 1u)
                    drained = mbar_wait(wfull0 + 8 * s, (a_par >> s) & 1u, nullptr, limit);
        }
        __syncwarp();
    } else if (warp == W_WARP) {
        // ----------------------------------------------------- W producer
        if (lane == 0) {
            const uint64_t pol_once = policy_evict_first();
            const uint64_t pol_reuse = policy_evict_last();  // also A: re-read by every n-tile
            Cursor<NQ> qc;
            Cursor<NBAR> bc;
            Cursor<WS> wc;
            Cursor<AS> ac;
            // the W slot's previous user (grouped GEMM: also m-tile 2's slot; the
            // A slot's previous user is one K-step older still)
            Cursor<NBAR> back = lag_cursor<WS>();
            uint32_t w_issued = 0, w_par = 0;
            bool ok = true;
            // Failure-detection test hook (off: stall < 0): CTA stall >> 40 arms
            // K-step (stall & 2^40-1) of its sequence but issues none of its
            // copies, so that K-step's full barrier never completes.
            const int64_t stall_step =
                (stall >= 0 && (stall >> 40) == blockIdx.x) ? (stall & ((int64_t{1} << 40) - 1)) : -1;
            int64_t kcount = 0;
            while (ok) {
                Unit U;
                const int got = q_pop<false>(qfull0, qempty0, ctl->q, qc, U, abort, limit);
                if (got <= 0) {
                    if (got < 0) fail(abort, status);
                    break;
                }
                const int nbox = U.bn / B_BOX;
                const uint64_t pol = U.shared_w ? pol_reuse : pol_once;
                // grouped GEMM: m-tiles 0, 1 to the A slot, m-tile 2 to the W slot
                const int a_lo = U.mpu < 2 ? U.mpu : 2;
                const uint32_t wtx = static_cast<uint32_t>(nbox * B_BOX_BYTES) +
                                     (!kGather && U.mpu > 2 ? static_cast<uint32_t>(A_BYTES) : 0u) +
                                     (kMx ? 1024u : 0u);
                const uint32_t atx = static_cast<uint32_t>(a_lo * A_BYTES);
                for (int ks = 0; ks < nk; ++ks) {
                    if (!mbar_wait(wempty0 + 8 * back.s, back.ph, abort, limit)) {
                        fail(abort, status);
                        ok = false;
                        break;
                    }
                    const uint32_t wfull = wfull0 + 8 * bc.s;
                    mbar_arrive_expect_tx(wfull, (kGather || kSplitA) ? wtx : wtx + atx);
                    const uint32_t wsl = sbase + wc.s * W_SLOT;
                    const bool stalled = kcount++ == stall_step;
                    for (int b = 0; b < nbox && !stalled; ++b) {
                        // bf16: 64 columns x 64 K rows (MN-major); FP8: 128 K codes x 64
                        // columns (K-major). Either way box b lands 8 KiB further.
                        if (kFp8)
                            tma_load_2d(wsl + b * B_BOX_BYTES, &wmap, 0,
                                        fp8_box_row(U.e, U.n0 / B_BOX + b, ks), wfull, pol);
                        else
                            tma_load_3d(wsl + b * B_BOX_BYTES, &wmap, U.n0 + b * B_BOX, ks * BKE,
                                        U.e, wfull, pol);
                    }
                    if (kMx && !stalled)  // W's block scales of this tile and K-step
                        bulk_g2s(wsl + MX_SFB_OFF,
                                 static_cast<const uint8_t*>(sw_) +
                                     ((static_cast<int64_t>(U.e) * ((De + MX_BN - 1) / MX_BN) +
                                       U.n0 / MX_BN) * nk + ks) * 1024,
                                 1024u, wfull, pol);
                    if (!stalled) {
                        w_issued |= 1u << bc.s;
                        w_par = (w_par & ~(1u << bc.s)) | (bc.ph << bc.s);
                    }
                    if (!kGather && !stalled) {  // rows past the expert's end are loaded but never stored
                        for (int mt = kSplitA ? 2 : 0; mt < U.mpu; ++mt)
                            tma_load_2d(a_tile(wc.s, ac.s, mt), &amap, ks * BKE, U.row0 + mt * BM,
                                        wfull, pol_reuse);
                    }
                    bc.next();
                    wc.next();
                    ac.next();
                    back.next();
                }
            }
            // Every copy this thread started must land before the CTA may exit
            // (the first wait that runs out ends the drain: see the A producer).
            bool drained = true;
            for (int s = 0; s < NBAR && drained; ++s)
                if ((w_issued >> s) & 1u)
                    drained = mbar_wait(wfull0 + 8 * s, (w_par >> s) & 1u, nullptr, limit);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ----------------------------------------------------------- MMA
        if (lane == 0) {
            Cursor<NQ> qc;
            Cursor<NBAR> bc;
            Cursor<WS> wc;
            Cursor<AS> ac;
            uint32_t acc_phase = 0;
            bool ok = true;
            // Descriptors of shared-memory address 0 (the address field holds
            // bytes >> 4, so an operand at byte offset o adds o >> 4).
            // A: K-major, rows 128 B apart, 8-row groups 1024 B apart; a K step
            // (16 bf16 or 32 FP8 elements) moves 32 B inside the swizzled row.
            // B (bf16): MN-major (W rows are N-contiguous), 64-column blocks
            // 8 KiB apart (LBO), 8-row K groups 1024 B apart (SBO); a K step of
            // 16 rows is 2 KiB. B (FP8): K-major like A.
            const uint64_t a_desc0 = sdesc_sw128(0, 16, 1024);
            const uint64_t b_desc0 = kFp8 ? sdesc_sw128(0, 16, 1024)
                                          : sdesc_sw128(0, B_BOX_BYTES, 1024);
            constexpr uint32_t b_step = kFp8 ? (32 >> 4) : ((UMMA_K * 128) >> 4);
            while (ok) {
                Unit U;
                const int got = q_pop<false>(qfull0, qempty0, ctl->q, qc, U, abort, limit);
                if (got <= 0) {
                    if (got < 0) fail(abort, status);
                    break;
                }
                if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort, limit)) {
                    fail(abort, status);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t idesc =
                    kFp8 ? idesc_e4m3_f32(BM, U.bn) : idesc_bf16_f32(BM, U.bn, true);
                const bool half = !kMx && half_last(U.mpu, U.rows);
                const uint32_t idesc_last =
                    !half ? idesc
                          : (kFp8 ? idesc_e4m3_f32(BM_HALF, U.bn)
                                  : idesc_bf16_f32(BM_HALF, U.bn, true));
                const int mpu = U.mpu;
                const uint32_t acc_stride = static_cast<uint32_t>(U.bn_max);
                for (int ks = 0; ks < nk; ++ks) {
                    if (!mbar_wait(wfull0 + 8 * bc.s, bc.ph, abort, limit)) {
                        fail(abort, status);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    // The gathered rows were written by cp.async (generic proxy);
                    // order them before the tensor cores' async-proxy reads.
                    fence_proxy_async_smem();
                    const uint64_t b_st = b_desc0 + ((sbase + wc.s * W_SLOT) >> 4);
                    // MX: this K-step's scales into TMEM buffer ac.s (its last
                    // reader, the K-step AS back, has completed: the rows
                    // of this K-step could only be gathered after it)
                    const uint32_t sft = tmem + MX_SF_TMEM + MX_SF_COLS * static_cast<uint32_t>(ac.s);
                    if (kMx) {
                        const uint32_t sfs = sbase + wc.s * W_SLOT + MX_SFB_OFF;
                        tmem_cp_32x128b_x4(sft + 8, sdesc_plain(sfs, 0, 128));
                        tmem_cp_32x128b_x4(sft + 12, sdesc_plain(sfs + 512, 0, 128));
                        for (int mt = 0; mt < mpu; ++mt)
                            tmem_cp_32x128b_x4(sft + 4 * mt,
                                               sdesc_plain(sfs + 1024 + 512 * mt, 0, 128));
                    }
                    for (int mt = 0; mt < mpu; ++mt) {
                        const uint64_t a_mt = a_desc0 + (a_tile(wc.s, ac.s, mt) >> 4);
                        const uint32_t id = mt == mpu - 1 ? idesc_last : idesc;
                        const uint32_t d = tmem + static_cast<uint32_t>(mt) * acc_stride;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {  // four K steps of 32 bytes per K-step
                            if (kMx)
                                mma_mx(d, a_mt + kk * (32 >> 4), b_st + kk * b_step,
                                       idesc_mx_e4m3(BM, U.bn, kk), sft + 4 * mt, sft + 8,
                                       (ks | kk) != 0 ? 1u : 0u);
                            else if (kFp8)
                                mma_f8(d, a_mt + kk * (32 >> 4), b_st + kk * b_step, id,
                                       (ks | kk) != 0 ? 1u : 0u);
                            else
                                mma_bf16(d, a_mt + kk * (32 >> 4), b_st + kk * b_step, id,
                                         (ks | kk) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(wempty0 + 8 * bc.s);
                    bc.next();
                    wc.next();
                    ac.next();
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
    } else if (warp < EPI_WARPS) {
        // ------------------------------------------------------ epilogue
        const int q = warp;  // TMEM lane quarter this warp may access (warps 0..3)
        const bool wide = (De % 16) == 0 && (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
        Cursor<NQ> qc;
        uint32_t acc_phase = 0;
        while (true) {
            Unit U;
            const int got = q_pop<true>(qfull0, qempty0, ctl->q, qc, U, abort, limit);
            if (got <= 0) {
                if (got < 0 && lane == 0) fail(abort, status);
                break;
            }
            // FP8: this lane's row scales (one per m-tile) and column scales
            // (one per 32 columns), loaded while the unit's MMAs still run.
            // Rows of m-tile mt in this warp's lane quarter: 32 from row
            // mt * BM + 32 q, or 16 from mt * BM + 16 q for an M = 64 last
            // m-tile (its lanes 0..15).
            const bool half = !kMx && half_last(U.mpu, U.rows);
            auto qrows = [&](int mt) { return (half && mt == U.mpu - 1) ? 16 : 32; };
            auto qrow0 = [&](int mt) { return mt * BM + qrows(mt) * q; };
            float rs_pre[MAX_MPU] = {1.0f, 1.0f, 1.0f};
            float cs_pre[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
            if (kFp8 && !kMx) {
#pragma unroll
                for (int mt = 0; mt < MAX_MPU; ++mt) {
                    const int r = qrow0(mt) + lane;
                    if (mt < U.mpu && lane < qrows(mt) && r < U.rows) {
                        if (kGather) {
                            const int f = __ldg(perm + U.row0 + r);
                            rs_pre[mt] = (f >= 0 && f < R) ? __ldg(sx + f / k) : 0.0f;
                        } else {
                            rs_pre[mt] = __ldg(sx + U.row0 + r);
                        }
                    }
                }
                const float* sw_u = sw + static_cast<int64_t>(U.e) * De;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int col = U.n0 + c * 32 + lane;
                    if (c * 32 < U.bn && col < De) cs_pre[c] = __ldg(sw_u + col);
                }
            }
            bool acc_ok = true;
            if (lane == 0)
                acc_ok = mbar_wait_backoff(acc_full, acc_phase, abort, limit, IDLE_SLEEP_NS);
            acc_ok = __shfl_sync(0xffffffffu, acc_ok ? 1 : 0, 0) != 0;
            __syncwarp();
            if (!acc_ok) {
                if (lane == 0) fail(abort, status);
                break;
            }
            tc_fence_after_sync();
            // Last m-tile with rows in this warp's quarter: TMEM is released
            // after its last load, before its last stores.
            int last_mt = -1;
            for (int mt = 0; mt < U.mpu; ++mt)
                if (qrow0(mt) < U.rows) last_mt = mt;
            bool released = false;
            for (int mt = 0; mt <= last_mt; ++mt) {
                const int rbase = qrow0(mt);
                if (rbase >= U.rows) continue;  // warp-uniform
                const int r = rbase + lane;
                const bool valid = lane < qrows(mt) && r < U.rows;
                uint16_t* orow = out + static_cast<int64_t>(U.row0 + r) * De;
                // FP8: this row's scale (its token's, or its own row's)
                const float rs = mt == 0 ? rs_pre[0] : (mt == 1 ? rs_pre[1] : rs_pre[2]);
                const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(mt * U.bn_max);
                for (int cc = 0; cc < U.bn / 32; cc += 2) {
                    // FP8: this lane's column scales (loaded before the accumulators were ready)
                    const float cs0 = cc == 0   ? cs_pre[0]
                                      : cc == 2 ? cs_pre[2]
                                      : cc == 4 ? cs_pre[4]
                                                : cs_pre[6];
                    const float cs1 = cc == 0   ? cs_pre[1]
                                      : cc == 2 ? cs_pre[3]
                                      : cc == 4 ? cs_pre[5]
                                                : cs_pre[7];
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(tbase + cc * 32, v0);
                    tmem_ld_32x32b_x32(tbase + cc * 32 + 32, v1);
                    tmem_wait_ld();
                    if (mt == last_mt && cc + 2 >= U.bn / 32) {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acc_empty);
                        released = true;
                    }
                    if (kFp8 && !kMx) {  // all lanes: the scales travel by shuffles
                        scale_chunk(v0, rs, cs0);
                        scale_chunk(v1, rs, cs1);
                    }
                    if (wide) {
                        store_rows_quad(out, static_cast<int64_t>(U.row0) + rbase,
                                        min(U.rows - rbase, qrows(mt)), De, v0, v1,
                                        U.n0 + cc * 32);
                    } else if (valid) {
                        store_row_chunk(orow, v0, U.n0 + cc * 32, De, false);
                        store_row_chunk(orow, v1, U.n0 + cc * 32 + 32, De, false);
                    }
                }
            }
            if (!released) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
            acc_phase ^= 1u;
        }
    }

    if (warp == SCHED_WARP) {
        // --------------------------------------------------------- scheduler
        // Walks the unit numbering for this CTA (units blockIdx.x, +gridDim.x,
        // ...) 32 experts at a time, one expert per lane, and queues each
        // unit's descriptor; a descriptor with e = -1 ends the list.
        const int nt256 = (De + 255) >> 8, nt128 = (De + 127) >> 7;
        const int ntmx = (De + MX_BN - 1) / MX_BN;
        int e0 = -32;
        int64_t before = 0, total = 0, cum = 0, units = 0;
        int lo = 0, rows = 0, mpu_max = 2, bn_max = 256, groups = 0, ntiles = 1;
        Cursor<NQ> qc;
        for (int64_t u = blockIdx.x;; u += gridDim.x) {
            bool have = false;
            while (true) {
                if (e0 >= 0 && u < before + total) {
                    have = true;
                    break;
                }
                if (e0 >= 0) before += total;
                e0 += 32;
                if (e0 >= E) break;
                const int e = e0 + lane;
                units = 0;
                rows = 0;
                if (e < E) {
                    lo = min(max(__ldg(offsets + e), 0), R);
                    const int hi = min(max(__ldg(offsets + e + 1), 0), R);
                    rows = max(hi, lo) - lo;
                    const int mt = (rows + BM - 1) / BM;
                    if (kMx) {
                        mpu_max = 2; bn_max = MX_BN; groups = (mt + 1) >> 1; ntiles = ntmx;
                    } else if (mt == 3) {
                        mpu_max = 3; bn_max = 128; groups = 1; ntiles = nt128;
                    } else {
                        mpu_max = 2; bn_max = 256; groups = (mt + 1) >> 1; ntiles = nt256;
                    }
                    units = static_cast<int64_t>(groups) * ntiles;
                }
                cum = units;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int64_t t = __shfl_up_sync(0xffffffffu, cum, d);
                    if (lane >= d) cum += t;
                }
                total = __shfl_sync(0xffffffffu, cum, 31);
            }
            int d[QWORDS] = {-1, 0, 0, 0, 0, 0, 0, 0};
            if (have) {
                const int64_t l = u - before;
                const int s = __ffs(__ballot_sync(0xffffffffu, l < cum)) - 1;
                const int s_lo = __shfl_sync(0xffffffffu, lo, s);
                const int s_rows = __shfl_sync(0xffffffffu, rows, s);
                const int s_mpu = __shfl_sync(0xffffffffu, mpu_max, s);
                const int s_bn = __shfl_sync(0xffffffffu, bn_max, s);
                const int s_groups = __shfl_sync(0xffffffffu, groups, s);
                const int s_nt = __shfl_sync(0xffffffffu, ntiles, s);
                const int64_t s_first = __shfl_sync(0xffffffffu, cum - units, s);
                const int li = static_cast<int>(l - s_first);
                const int g = li / s_nt, n = li - g * s_nt;
                d[0] = e0 + s;
                d[1] = s_lo + g * (s_mpu * BM);
                d[2] = min(s_mpu * BM, s_rows - g * (s_mpu * BM));
                d[3] = (d[2] + BM - 1) / BM;
                d[4] = n * s_bn;
                d[5] = min(s_bn, (De - d[4] + B_BOX - 1) / B_BOX * B_BOX);
                d[6] = s_bn;
                d[7] = s_groups > 1 ? 1 : 0;
            }
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait_backoff(qempty0 + 8 * qc.s, qc.ph ^ 1u, abort, limit,
                                       IDLE_SLEEP_NS);
                if (ok) {
#pragma unroll
                    for (int i = 0; i < QWORDS; ++i) ctl->q[qc.s][i] = d[i];
                    mbar_arrive(qfull0 + 8 * qc.s);
                } else {
                    fail(abort, status);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            qc.next();
            if (!have || !ok) break;
        }
    }
    // (every role comes here when done)
    tc_fence_before_sync();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace dg

// ------------------------------------------------------------------ host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<int64_t> g_debug_stall{-1};
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

// Tensor map of the expert weights. bf16 W [E, D, De]: a 3-D map {De, D, E}
// with 64 x 64 boxes. FP8 codes in the blocked layout: a [rows, 128] byte
// matrix of 64-row boxes (rows = E * ceil(De/64) * ceil(D/128) * 64). Both
// with 128-byte swizzle; out-of-range boxes read zeros.
int make_w_map(bool fp8, const void* W, int32_t D, int32_t E, int32_t De, CUtensorMap* wmap) {
    using namespace dg;
    auto enc = encoder();
    if (!enc) return PK_ERR_CUDA;
    if (fp8) {
        const uint64_t rows = static_cast<uint64_t>(E) * ((De + B_BOX - 1) / B_BOX) *
                              ((D + ROW_BYTES - 1) / ROW_BYTES) * B_BOX;
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(ROW_BYTES), static_cast<cuuint64_t>(rows)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(ROW_BYTES)};
        cuuint32_t box[2] = {ROW_BYTES, B_BOX};
        cuuint32_t es[2] = {1, 1};
        if (enc(wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), dims, strides, box,
                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PK_ERR_UNSUPPORTED;
    } else {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(De), static_cast<cuuint64_t>(D),
                              static_cast<cuuint64_t>(E)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(De) * 2,
                                 static_cast<cuuint64_t>(D) * static_cast<cuuint64_t>(De) * 2};
        cuuint32_t box[3] = {B_BOX, BK, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PK_ERR_UNSUPPORTED;
    }
    return PK_OK;
}

namespace {

// Builds the tensor maps and launches one instantiation. A is x (gathered
// through perm) or, without gather, the [T, D] matrix of expert-sorted rows.
// fp8: x and W are E4M3 codes (W blocked, see pk_moe_fp8_weight_bytes) with
// scales sx [T], sw [E, De] (fp32), or with mx, E8M0 block scales (sx the
// rows' bytes [T, D / 32], sw the weights' scale pieces).
int launch_common(bool gather, bool fp8, const void* A, const void* sx, const int32_t* perm,
                  const int32_t* offsets, const void* W, const void* sw, int32_t T, int32_t k,
                  int32_t D, int32_t E, int32_t De, uint16_t* out, int32_t* status,
                  cudaStream_t stream, uint64_t wait_limit_ns, bool mx = false) {
    const int64_t stall = g_debug_stall.load(std::memory_order_relaxed);
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
            // every instantiation launch_common can launch
            const void* kernels[] = {
                reinterpret_cast<const void*>(k_dispatch_gemm<true, false>),
                reinterpret_cast<const void*>(k_dispatch_gemm<true, false, false, true>),
                reinterpret_cast<const void*>(k_dispatch_gemm<true, true>),
                reinterpret_cast<const void*>(k_dispatch_gemm<true, true, false, true>),
                reinterpret_cast<const void*>(k_dispatch_gemm<true, true, true>),
                reinterpret_cast<const void*>(k_dispatch_gemm<true, true, true, true>),
                reinterpret_cast<const void*>(k_dispatch_gemm<false, false, false, true>),
                reinterpret_cast<const void*>(k_dispatch_gemm<false, true, false, true>)};
            for (const void* kern : kernels)
                if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES) != cudaSuccess)
                    return PK_ERR_CUDA;
            di.attr_set = true;
        }
        sms = di.sms;
    }

    CUtensorMap wmap, amap;
    const int rc = make_w_map(fp8, W, D, E, De, &wmap);
    if (rc != PK_OK) return rc;
    if (gather) {
        amap = wmap;  // unused
    } else {
        // A [T, D] row-major, boxes of 128 bytes (64 bf16 or 128 E4M3 codes) x 128
        // rows, 128-byte swizzle
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * (fp8 ? 1 : 2)};
        cuuint32_t box[2] = {fp8 ? static_cast<cuuint32_t>(ROW_BYTES) : static_cast<cuuint32_t>(BK),
                             static_cast<cuuint32_t>(BM)};
        cuuint32_t es[2] = {1, 1};
        if (enc(&amap, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                const_cast<void*>(A), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PK_ERR_UNSUPPORTED;
    }
    const uint8_t* a8 = static_cast<const uint8_t*>(A);
    // gathered rows that stay in L2 (x small): the deep W ring
    const bool deep = gather && static_cast<int64_t>(T) * D * (fp8 ? 1 : 2) <= DEEP_W_MAX_X_BYTES;
    if (mx && deep)
        k_dispatch_gemm<true, true, true, true><<<sms, THREADS, SMEM_BYTES, stream>>>(
            wmap, amap, a8, sx, sw, perm, offsets, out, T, k, D, E, De, status, wait_limit_ns, stall);
    else if (mx)
        k_dispatch_gemm<true, true, true><<<sms, THREADS, SMEM_BYTES, stream>>>(
            wmap, amap, a8, sx, sw, perm, offsets, out, T, k, D, E, De, status, wait_limit_ns, stall);
    else if (fp8 && gather && deep)
        k_dispatch_gemm<true, true, false, true><<<sms, THREADS, SMEM_BYTES, stream>>>(
            wmap, amap, a8, sx, sw, perm, offsets, out, T, k, D, E, De, status, wait_limit_ns, stall);
    else if (fp8 && gather)
        k_dispatch_gemm<true, true><<<sms, THREADS, SMEM_BYTES, stream>>>(
            wmap, amap, a8, sx, sw, perm, offsets, out, T, k, D, E, De, status, wait_limit_ns, stall);
    else if (fp8)
        k_dispatch_gemm<false, true, false, true><<<sms, THREADS, SMEM_BYTES, stream>>>(
            wmap, amap, a8, sx, sw, nullptr, offsets, out, T, k, D, E, De, status, wait_limit_ns, stall);
    else if (gather && deep)
        k_dispatch_gemm<true, false, false, true><<<sms, THREADS, SMEM_BYTES, stream>>>(
            wmap, amap, a8, nullptr, nullptr, perm, offsets, out, T, k, D, E, De, status,
            wait_limit_ns, stall);
    else if (gather)
        k_dispatch_gemm<true, false><<<sms, THREADS, SMEM_BYTES, stream>>>(
            wmap, amap, a8, nullptr, nullptr, perm, offsets, out, T, k, D, E, De, status,
            wait_limit_ns, stall);
    else
        k_dispatch_gemm<false, false, false, true><<<sms, THREADS, SMEM_BYTES, stream>>>(
            wmap, amap, a8, nullptr, nullptr, perm, offsets, out, T, k, D, E, De, status,
            wait_limit_ns, stall);
    return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

}  // namespace

int launch_dispatch_gemm_single(const uint16_t* x, const int32_t* perm, const int32_t* offsets,
                                const uint16_t* W, int32_t T, int32_t k, int32_t D, int32_t E,
                                int32_t De, uint16_t* out, int32_t* status, cudaStream_t stream,
                                uint64_t wait_limit_ns) {
    return launch_common(true, false, x, nullptr, perm, offsets, W, nullptr, T, k, D, E, De, out,
                         status, stream, wait_limit_ns);
}

int launch_dispatch_gemm_fp8_single(const uint8_t* xq, const float* sx, const int32_t* perm,
                                    const int32_t* offsets, const uint8_t* wq, const float* sw,
                                    int32_t T, int32_t k, int32_t D, int32_t E, int32_t De,
                                    uint16_t* out, int32_t* status, cudaStream_t stream,
                                    uint64_t wait_limit_ns) {
    return launch_common(true, true, xq, sx, perm, offsets, wq, sw, T, k, D, E, De, out, status,
                         stream, wait_limit_ns);
}

int launch_dispatch_gemm_mx(const uint8_t* xq, const uint8_t* sx, const int32_t* perm,
                            const int32_t* offsets, const uint8_t* wq, const uint8_t* swb,
                            int32_t T, int32_t k, int32_t D, int32_t E, int32_t De, uint16_t* out,
                            int32_t* status, cudaStream_t stream, uint64_t wait_limit_ns) {
    return launch_common(true, true, xq, sx, perm, offsets, wq, swb, T, k, D, E, De, out, status,
                         stream, wait_limit_ns, true);
}

void set_debug_stall(int32_t cta, int64_t kstep) {
    g_debug_stall.store(cta >= 0 && kstep >= 0 && kstep < (int64_t{1} << 40)
                            ? (static_cast<int64_t>(cta) << 40) | kstep
                            : -1,
                        std::memory_order_relaxed);
}

int launch_grouped_gemm(const uint16_t* A, const int32_t* offsets, const uint16_t* W, int32_t R,
                        int32_t K, int32_t N, int32_t E, uint16_t* out, int32_t* status,
                        cudaStream_t stream, uint64_t wait_limit_ns) {
    return launch_common(false, false, A, nullptr, nullptr, offsets, W, nullptr, R, 1, K, E, N,
                         out, status, stream, wait_limit_ns);
}

int launch_grouped_gemm_fp8(const uint8_t* Aq, const float* sa, const int32_t* offsets,
                            const uint8_t* wq, const float* sw, int32_t R, int32_t K, int32_t N,
                            int32_t E, uint16_t* out, int32_t* status, cudaStream_t stream,
                            uint64_t wait_limit_ns) {
    return launch_common(false, true, Aq, sa, nullptr, offsets, wq, sw, R, 1, K, E, N, out, status,
                         stream, wait_limit_ns);
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
