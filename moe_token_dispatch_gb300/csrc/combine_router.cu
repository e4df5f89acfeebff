// The steps on either side of the dispatch + expert GEMM of "Loads and Loads
// of Fluffy Kittens" ("Key claims", Fig. 17: top_k=8, num_experts=256):
//
//   k_router_topk  the router's selection: for every token, the k experts
//                  with the largest logits (largest first, equal logits to
//                  the lower expert) and gates = softmax over those k logits.
//   k_combine      un-permute and weight the expert outputs back into token
//                  order: y[t, :] = sum_s gates[t, s] * src[inv_perm[t*k+s], :],
//                  fp32 accumulation in increasing s, one bf16 rounding.
//
// Both are memory-bound streaming kernels: one warp per token (router) or per
// (token, 512-column chunk) (combine), 16-byte vector loads, grids sized to a
// few resident warps per SM sub-partition.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pk_internal.h"
#include "pk_ptx.cuh"

namespace pk {

// ------------------------------------------------------------------ router
// Unsigned key with the order of the float values (finite or infinite, not
// NaN): negative floats have their bits inverted, the rest their sign bit set;
// -0 is mapped like +0, so keys of equal values are equal. Non-negative keys
// start at 0x80000000, so 0 is below every real value.
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// PER = logits held per lane (E <= 32 * PER), a power of two so that the
// selection loops are fully unrolled for the common expert counts.
template <int PER>
__global__ void __launch_bounds__(256)
    k_router_topk(const float* __restrict__ logits, int32_t T, int32_t E, int32_t k,
                  int32_t* __restrict__ topk, float* __restrict__ gates) {
    constexpr int kNone = 0x7fffffff;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = warp0; t < T; t += nwarps) {
        const float* row = logits + t * E;
        float v[PER];
        uint32_t avail = 0;  // bit i: entry i of this lane exists and is not taken
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = i * 32 + lane;
            v[i] = e < E ? __ldg(row + e) : -INFINITY;
            if (e < E) avail |= 1u << i;
        }
        float my_val = -INFINITY;
        int my_idx = 0;
        for (int s = 0; s < k; ++s) {
            // this lane's best available entry; e grows with i, so replacing
            // only on a strictly larger value keeps the lowest index among equals
            float bv = -INFINITY;
            int bi = kNone;
#pragma unroll
            for (int i = 0; i < PER; ++i)
                if (((avail >> i) & 1u) && (bi == kNone || v[i] > bv)) {
                    bv = v[i];
                    bi = i * 32 + lane;
                }
            // warp arg-max in two reductions: the largest value (as an
            // order-preserving integer key, -0 folded into +0 so that equal
            // logits compare equal), then the lowest index holding it
            const uint32_t key = bi == kNone ? 0u : order_key(bv);
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
            const int wi = static_cast<int>(__reduce_min_sync(
                0xffffffffu, key == kmax && bi != kNone ? static_cast<uint32_t>(bi) : 0xffffffffu));
            const float wv = __shfl_sync(0xffffffffu, bv, wi & 31);
            if ((wi & 31) == lane) avail &= ~(1u << (wi >> 5));
            if (lane == s) {
                my_val = wv;
                my_idx = wi;
            }
        }
        // softmax over the selected logits, shifted by the largest (slot 0)
        const float m = __shfl_sync(0xffffffffu, my_val, 0);
        const float ex = lane < k ? expf(my_val - m) : 0.0f;
        float z = ex;
        for (int d = 16; d > 0; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
        if (lane < k) {
            topk[t * k + lane] = my_idx;
            if (gates) gates[t * k + lane] = ex / z;
        }
    }
}

// ----------------------------------------------------------------- combine
constexpr int kCombineSlotBatch = 8;  // source rows loaded before they are summed

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// VEC: 16-byte vectors per lane per source row; a warp covers 256 * VEC
// columns of a token (each load instruction of the warp 512 contiguous bytes).
template <int VEC>
__global__ void __launch_bounds__(256)
    k_combine(const uint16_t* __restrict__ src, const int32_t* __restrict__ inv_perm,
              const float* __restrict__ gates, int32_t T, int32_t k, int32_t C,
              uint16_t* __restrict__ y, int32_t* status) {
    constexpr int kCols = 256 * VEC;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int chunks = (C + kCols - 1) / kCols;
    const int64_t items = static_cast<int64_t>(T) * chunks;
    const int64_t R = static_cast<int64_t>(T) * k;
    bool bad = false;
    for (int64_t it = warp0; it < items; it += nwarps) {
        const int64_t t = it / chunks;
        const int cbase = static_cast<int>(it - t * chunks) * kCols + lane * 8;
        float acc[VEC][8];
#pragma unroll
        for (int u = 0; u < VEC; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
        for (int s0 = 0; s0 < k; s0 += kCombineSlotBatch) {
            uint4 v[kCombineSlotBatch][VEC];
            float g[kCombineSlotBatch];
#pragma unroll
            for (int i = 0; i < kCombineSlotBatch; ++i) {
                const int s = s0 + i;
                g[i] = 0.0f;
#pragma unroll
                for (int u = 0; u < VEC; ++u) v[i][u] = make_uint4(0, 0, 0, 0);
                if (s < k) {
                    int64_t j = __ldg(inv_perm + t * k + s);
                    if (j < 0 || j >= R) {
                        bad = true;
                        j = 0;
                    }
                    g[i] = gates ? __ldg(gates + t * k + s) : 1.0f;
#pragma unroll
                    for (int u = 0; u < VEC; ++u)
                        if (cbase + u * 256 < C) v[i][u] = ld_nc_v4(src + j * C + cbase + u * 256);
                }
            }
#pragma unroll
            for (int i = 0; i < kCombineSlotBatch; ++i) {
                if (s0 + i < k) {
#pragma unroll
                    for (int u = 0; u < VEC; ++u) {
                        const uint32_t w[4] = {v[i][u].x, v[i][u].y, v[i][u].z, v[i][u].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            acc[u][2 * h] = fmaf(g[i], __uint_as_float(w[h] << 16), acc[u][2 * h]);
                            acc[u][2 * h + 1] = fmaf(g[i], __uint_as_float(w[h] & 0xffff0000u),
                                                     acc[u][2 * h + 1]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < VEC; ++u) {
            if (cbase + u * 256 < C) {
                uint4 o;
                uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[u][2 * h], acc[u][2 * h + 1]);
                    ow[h] = *reinterpret_cast<uint32_t*>(&b2);
                }
                *reinterpret_cast<uint4*>(y + t * C + cbase + u * 256) = o;
            }
        }
    }
    if (bad) report(status, PK_ERR_BAD_INDEX);
}

namespace {
int g_sms_cr[64] = {0};

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!g_sms_cr[dev]) cudaDeviceGetAttribute(&g_sms_cr[dev], cudaDevAttrMultiProcessorCount, dev);
    return g_sms_cr[dev];
}
}  // namespace

cudaError_t launch_router_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                               int32_t* topk, float* gates, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int sms = sm_count();
    if (!sms) return cudaErrorInvalidDevice;
    const int64_t blocks = (static_cast<int64_t>(T) + 7) / 8;
    const int grid = static_cast<int>(blocks < sms * 16 ? blocks : sms * 16);
    const int per = (E + 31) / 32;
    if (per <= 1)
        k_router_topk<1><<<grid, 256, 0, stream>>>(logits, T, E, k, topk, gates);
    else if (per <= 2)
        k_router_topk<2><<<grid, 256, 0, stream>>>(logits, T, E, k, topk, gates);
    else if (per <= 4)
        k_router_topk<4><<<grid, 256, 0, stream>>>(logits, T, E, k, topk, gates);
    else if (per <= 8)
        k_router_topk<8><<<grid, 256, 0, stream>>>(logits, T, E, k, topk, gates);
    else if (per <= 16)
        k_router_topk<16><<<grid, 256, 0, stream>>>(logits, T, E, k, topk, gates);
    else
        k_router_topk<32><<<grid, 256, 0, stream>>>(logits, T, E, k, topk, gates);
    return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* src, const int32_t* inv_perm, const float* gates,
                           int32_t T, int32_t k, int32_t C, uint16_t* y, int32_t* status,
                           cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int sms = sm_count();
    if (!sms) return cudaErrorInvalidDevice;
    // two vectors per lane: 1 KiB of each source row per warp (95 % of the HBM
    // copy rate at ep against 85 % with 512 bytes)
    constexpr int vec = 2;
    const int64_t items = static_cast<int64_t>(T) * ((C + 256 * vec - 1) / (256 * vec));
    const int64_t blocks = (items + 7) / 8;
    const int grid = static_cast<int>(blocks < sms * 8 ? blocks : sms * 8);
    k_combine<vec><<<grid, 256, 0, stream>>>(src, inv_perm, gates, T, k, C, y, status);
    return cudaGetLastError();
}

}  // namespace pk
