// Inline-PTX building blocks for sm_103a: shared-memory barriers, TMA bulk
// tensor copies and L2 prefetches, tcgen05 tensor-core MMAs with
// accumulators in tensor memory (TMEM), and the shared-memory matrix
// descriptors they read. Written from the PTX ISA (tcgen05, cp.async.bulk.tensor,
// mbarrier chapters); no library code.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace pk {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lane_id() {
    uint32_t l;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
    return l;
}

// Records the first device-side error in *status (nullable).
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------ programmatic dependent launch
// A kernel launched with programmatic stream serialisation may start before
// the kernel ahead of it in the stream has finished. grid_dep_wait() returns
// once that kernel has completed and its writes are visible (at once when the
// launch had no such dependency); grid_dep_release() lets the next kernel of
// the stream start launching its blocks.
__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_release() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test_parity(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits until the phase with the given parity has completed. Gives up (and
// returns false) when *abort (nullable) becomes non-zero or after limit_ns
// nanoseconds of the global timer. A second bound of 4 SM cycles per
// nanosecond of the limit ends the wait even if the timer stood still.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                          uint64_t limit_ns) {
    if (mbar_test_parity(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const long long c0 = clock64();
    const long long cmax =
        limit_ns < (1ull << 60) ? static_cast<long long>(limit_ns * 4) : (1ll << 62);
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_test_parity(bar, parity)) return true;
        if (abort && *abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
        if (clock64() - c0 > cmax) return false;
    }
}

// mbar_wait for waits that usually last many microseconds (a role idle for
// a whole work unit): between tests the thread sleeps about sleep_ns, so that
// the idle warps draw less power on a power-capped GPU. Same limits.
__device__ __forceinline__ bool mbar_wait_backoff(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort, uint64_t limit_ns,
                                                  uint32_t sleep_ns) {
    if (mbar_test_parity(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const long long c0 = clock64();
    const long long cmax =
        limit_ns < (1ull << 60) ? static_cast<long long>(limit_ns * 4) : (1ll << 62);
    while (true) {
        if (mbar_test_parity(bar, parity)) return true;
        __nanosleep(sleep_ns);
        if (abort && *abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
        if (clock64() - c0 > cmax) return false;
    }
}

// ------------------------------------------------------------------ TMA
// Tiled 3-D load of one box into shared memory; completion is counted in
// bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// Brings one box of a 3-D tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map),
                 "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// L2 eviction-priority policies for the cache_hint operand.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// --------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Each thread of the warp reads 32 consecutive fp32 columns of its own TMEM
// lane (lane = warp's lane quarter * 32 + lane id).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format) for a 128-byte-swizzled
// operand: start address, leading/stride byte offsets (both >> 4), the
// descriptor version bits (46..47 = 1) and swizzle mode 2 (128 B) in bits
// 61..63. Base offset 0: every swizzle atom starts on a 1024-byte boundary.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator (bits 4..5 = 1),
// A and B bf16 (bits 7..9 = 1, 10..12 = 1), A K-major (bit 15 = 0), B major
// mode in bit 16 (1 = MN-major), N >> 3 in bits 17..22, M >> 4 in bits 24..28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace pk

namespace pk {

// ------------------------------------------------- cp.async (LSU path)
// 16-byte global -> shared copy through L2 only; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes,
                                            uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst),
                 "l"(src), "r"(src_bytes), "l"(policy)
                 : "memory");
}
// The barrier counts one arrival (already included in its expected count)
// once every cp.async this thread issued so far has completed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
// Orders generic-proxy shared-memory writes that this thread has observed
// (its own, or others' through a barrier it waited on) before its later
// async-proxy operations (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace pk

namespace pk {

// ------------------------------------------------------- thread-block cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
}

}  // namespace pk

namespace pk {
// Tiled 2-D load of one box into shared memory; completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}
}  // namespace pk

namespace pk {
// D[tmem] (+)= A * B with 8-bit float inputs (E4M3 or E5M2 per the
// instruction descriptor), fp32 accumulate, no block scaling.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor for kind::f8f6f4 with E4M3 A and B (format code 0 in
// bits 7..9 and 10..12), fp32 accumulator (bits 4..5 = 1), both operands
// K-major, N >> 3 in bits 17..22, M >> 4 in bits 24..28.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
}  // namespace pk

namespace pk {
// ------------------------------------------------ CTA-pair (cta_group::2) forms
// A pair of CTAs (ranks 0 and 1 of a 2-CTA cluster) shares one tensor-core
// operation: rank 0 issues tcgen05.mma.cta_group::2 with M = 256; A's rows
// 0..127 come from rank 0's shared memory and rows 128..255 from rank 1's,
// B's columns are split in halves the same way (N/2 columns in each CTA, at
// the same shared-memory offset as the descriptor), and each CTA's TMEM lanes
// 0..127 receive its own 128 rows of D for all N columns. Every tcgen05
// instruction of such a kernel uses cta_group::2; allocation is collective
// (one warp in each CTA, same column address in both).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void mma_pair_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_pair_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on the barrier at offset `bar` in every CTA of `cta_mask` when
// all tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"(cta_mask)
        : "memory");
}
// Arrive (release at cluster scope) on a barrier of another CTA of the
// cluster; `bar_cluster` is its shared::cluster address (map_to_cta).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}
__device__ __forceinline__ bool mbar_test_parity_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// mbar_wait for barriers that other CTAs arrive on (acquire at cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort, uint64_t limit_ns) {
    if (mbar_test_parity_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const long long c0 = clock64();
    const long long cmax =
        limit_ns < (1ull << 60) ? static_cast<long long>(limit_ns * 4) : (1ll << 62);
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_test_parity_cluster(bar, parity)) return true;
        if (abort && *abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
        if (clock64() - c0 > cmax) return false;
    }
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr_cluster, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr_cluster), "r"(v) : "memory");
}
}  // namespace pk

namespace pk {
// ------------------------------------------------------- microscaled FP8 (MX)
// D[tmem] (+)= (A * 2^sa) * (B * 2^sb): E4M3 operands, one E8M0 scale per 32
// K-elements of every row of A and every column of B (kind::mxf8f6f4,
// scale_vec::1X), fp32 accumulate. The scales are read from TMEM: for row m
// of A from lane m, column sa_tmem + m / 32; for column n of B, by the rows
// of lane quarter q, from lane 32 q + n % 32, column sb_tmem + n / 32. Each
// 32-bit cell holds four scale bytes; the instruction descriptor's scale ids
// pick the byte (measured on GB300 with patterned scales).
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t sa_tmem, uint32_t sb_tmem,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sa_tmem), "r"(sb_tmem), "r"(accumulate)
        : "memory");
}

// Instruction descriptor for kind::mxf8f6f4 with E4M3 A and B (format 0 in bits
// 7..9 and 10..12), both K-major, E8M0 scales (bit 23), N >> 3 in bits 17..22,
// M >> 4 in bits 24..28, the byte of B's and A's scale cells in bits 4..5 and
// 29..30.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int M, int N, int sf_id) {
    return (static_cast<uint32_t>(sf_id & 3) << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
           (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) |
           (static_cast<uint32_t>(sf_id & 3) << 29);
}

// Shared-memory matrix descriptor without swizzle: start address, leading and
// stride byte offsets (both >> 4), descriptor version 1 in bits 46..47.
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// Copies a 32-row x 16-byte block of shared memory (rows 16 bytes apart; a
// plain descriptor with 128-byte stride between 8-row groups) into TMEM
// lanes 0..31, columns taddr .. taddr+3, and the same into the other three
// lane quarters. Ordered with this thread's later tcgen05.mma.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// Bulk copy global -> shared memory of `bytes` (multiple of 16, both
// addresses 16-byte aligned), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 4-byte global -> shared copy through the LSU path (tracked by the thread's
// cp.async arrivals like cp_async_16).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
}  // namespace pk
