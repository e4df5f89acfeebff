// E4M3 quantisation for the FP8 expert GEMM, one float32 scale per vector:
//   amax = max |v|,  inv = 448 / amax,  code = E4M3_rn_satfinite(v * inv),
//   scale = amax / 448
// with IEEE float32 division and multiplication, so the codes are a pure
// function of the bf16 inputs. When amax == 0 or 448 / amax overflows (amax
// below about 1.3e-36), inv = scale = 1 and every code is zero. Inputs are
// finite.
//   k_quant_rows_reg    activations x [T, D] -> codes [T, D] + scales [T]
//                       (one block per row held in registers, x read once;
//                       D <= 8192), else
//   k_quant_rows        the same with one warp per row and two passes.
//   k_col_amax,
//   k_col_convert,
//   k_col_scale         weights W [E, D, N] -> codes in the blocked layout
//                       the FP8 GEMM reads (each 64-column x 128-code block
//                       contiguous, K-major inside: column n's codes d of one
//                       block form one 128-byte row) + scales [E, N]; done
//                       once per weight set, not per step.
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pk_internal.h"

namespace pk {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// 448 / amax, or 1 where that is not a finite number (amax == 0 or tiny)
__device__ __forceinline__ float inv_scale(float amax) {
    const float r = __fdiv_rn(448.0f, amax);
    return (amax > 0.0f && isfinite(r)) ? r : 1.0f;
}
__device__ __forceinline__ float scale_of(float amax) {
    return (amax > 0.0f && isfinite(__fdiv_rn(448.0f, amax))) ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    return static_cast<uint16_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__global__ void __launch_bounds__(256)
    k_quant_rows(const uint16_t* __restrict__ x, int32_t T, int32_t D, uint8_t* __restrict__ q,
                 float* __restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = warp0; t < T; t += nwarps) {
        const uint16_t* row = x + t * D;
        float amax = 0.0f;
        for (int c = lane * 8; c < D; c += 256) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
                amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(w[h] & 0xffffu)),
                                         fabsf(bf16_bits_to_f32(w[h] >> 16))));
        }
        for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        const float inv = inv_scale(amax);
        if (lane == 0) scale[t] = scale_of(amax);
        uint8_t* qrow = q + t * D;
        for (int c = lane * 8; c < D; c += 256) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t out[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint16_t a = e4m3x2(__fmul_rn(bf16_bits_to_f32(w[2 * h] & 0xffffu), inv),
                                          __fmul_rn(bf16_bits_to_f32(w[2 * h] >> 16), inv));
                const uint16_t b = e4m3x2(__fmul_rn(bf16_bits_to_f32(w[2 * h + 1] & 0xffffu), inv),
                                          __fmul_rn(bf16_bits_to_f32(w[2 * h + 1] >> 16), inv));
                out[h] = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
            }
            *reinterpret_cast<uint2*>(qrow + c) = make_uint2(out[0], out[1]);
        }
    }
}

// One block of kRowThreads per row, the row held in registers (VPT 16-byte
// vectors per thread, D <= kRowThreads * 8 * VPT): x is read once; the
// block's amax comes from warp shuffles and one shared-memory step.
constexpr int kRowThreads = 256;
template <int VPT>
__global__ void __launch_bounds__(kRowThreads)
    k_quant_rows_reg(const uint16_t* __restrict__ x, int32_t T, int32_t D,
                     uint8_t* __restrict__ q, float* __restrict__ scale) {
    __shared__ float wmax[kRowThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const uint16_t* row = x + t * D;
        uint4 v[VPT];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = (i * kRowThreads + threadIdx.x) * 8;
            v[i] = c < D ? *reinterpret_cast<const uint4*>(row + c) : make_uint4(0, 0, 0, 0);
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
                amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(w[h] & 0xffffu)),
                                         fabsf(bf16_bits_to_f32(w[h] >> 16))));
        }
        for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        if (lane == 0) wmax[warp] = amax;
        __syncthreads();
        amax = wmax[0];
#pragma unroll
        for (int w = 1; w < kRowThreads / 32; ++w) amax = fmaxf(amax, wmax[w]);
        __syncthreads();  // wmax is rewritten by the next row
        const float inv = inv_scale(amax);
        if (threadIdx.x == 0) scale[t] = scale_of(amax);
        uint8_t* qrow = q + t * D;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = (i * kRowThreads + threadIdx.x) * 8;
            if (c < D) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t o[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint16_t a = e4m3x2(__fmul_rn(bf16_bits_to_f32(w[2 * h] & 0xffffu), inv),
                                              __fmul_rn(bf16_bits_to_f32(w[2 * h] >> 16), inv));
                    const uint16_t b = e4m3x2(__fmul_rn(bf16_bits_to_f32(w[2 * h + 1] & 0xffffu), inv),
                                              __fmul_rn(bf16_bits_to_f32(w[2 * h + 1] >> 16), inv));
                    o[h] = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
                }
                *reinterpret_cast<uint2*>(qrow + c) = make_uint2(o[0], o[1]);
            }
        }
    }
}

// amax of every column of W[e] into amax_out[e, n]
__global__ void __launch_bounds__(256)
    k_col_amax(const uint16_t* __restrict__ W, int32_t D, int32_t N, float* __restrict__ amax_out) {
    const int e = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    const uint16_t* col = W + static_cast<int64_t>(e) * D * N + n;
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) amax = fmaxf(amax, fabsf(bf16_bits_to_f32(col[static_cast<int64_t>(d) * N])));
    amax_out[static_cast<int64_t>(e) * N + n] = amax;
}

// codes of a 32 (d) x 32 (n) tile, written transposed into the blocked
// layout: code (e, n, d) at byte ((((e * NB + n / 64) * KB + d / 128) * 64 +
// n % 64) * 128 + d % 128, NB = ceil(N / 64), KB = ceil(D / 128)
__global__ void __launch_bounds__(256)
    k_col_convert(const uint16_t* __restrict__ W, int32_t D, int32_t N,
                  const float* __restrict__ amax, uint8_t* __restrict__ q) {
    const int64_t NB = (N + 63) / 64, KB = (D + 127) / 128;
    __shared__ uint8_t tile[32][33];
    const int e = blockIdx.z;
    const int n0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const int n = n0 + tx;
    float inv = 1.0f;
    if (n < N) {
        inv = inv_scale(amax[static_cast<int64_t>(e) * N + n]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int d = d0 + ty + 8 * i;
        uint8_t c = 0;
        if (n < N && d < D) {
            const float v = bf16_bits_to_f32(W[(static_cast<int64_t>(e) * D + d) * N + n]);
            c = static_cast<uint8_t>(e4m3x2(__fmul_rn(v, inv), 0.0f) & 0xffu);
        }
        tile[ty + 8 * i][tx] = c;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int nn = n0 + ty + 8 * i, d = d0 + tx;
        if (nn < N && d < D) {
            const int64_t row = ((e * NB + nn / 64) * KB + d / 128) * 64 + nn % 64;
            q[row * 128 + d % 128] = tile[tx][ty + 8 * i];
        }
    }
}

__global__ void k_col_scale(float* __restrict__ s, int64_t n) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) {
        s[i] = scale_of(s[i]);
    }
}

cudaError_t launch_quant_rows(const uint16_t* x, int32_t T, int32_t D, uint8_t* q, float* scale,
                              cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    if (D <= kRowThreads * 8 * 4) {  // the row fits the block's registers: one read of x
        const int grid = static_cast<int>(T < sms * 64 ? T : sms * 64);
        if (D <= kRowThreads * 8 * 2)
            k_quant_rows_reg<2><<<grid, kRowThreads, 0, stream>>>(x, T, D, q, scale);
        else
            k_quant_rows_reg<4><<<grid, kRowThreads, 0, stream>>>(x, T, D, q, scale);
        return cudaGetLastError();
    }
    const int64_t blocks = (static_cast<int64_t>(T) + 7) / 8;
    const int grid = static_cast<int>(blocks < sms * 16 ? blocks : sms * 16);
    k_quant_rows<<<grid, 256, 0, stream>>>(x, T, D, q, scale);
    return cudaGetLastError();
}

cudaError_t launch_quant_cols(const uint16_t* W, int32_t E, int32_t D, int32_t N, uint8_t* q,
                              float* scale, cudaStream_t stream) {
    // padding of the blocks past D and N reads as code 0
    const int64_t bytes = static_cast<int64_t>(E) * ((N + 63) / 64) * ((D + 127) / 128) * 8192;
    cudaError_t err = cudaMemsetAsync(q, 0, static_cast<size_t>(bytes), stream);
    if (err != cudaSuccess) return err;
    // scale holds each column's amax until the last kernel turns it into the scale
    k_col_amax<<<dim3((N + 255) / 256, E), 256, 0, stream>>>(W, D, N, scale);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    k_col_convert<<<dim3((N + 31) / 32, (D + 31) / 32, E), 256, 0, stream>>>(W, D, N, scale, q);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int64_t n = static_cast<int64_t>(E) * N;
    k_col_scale<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(scale, n);
    return cudaGetLastError();
}

}  // namespace pk
